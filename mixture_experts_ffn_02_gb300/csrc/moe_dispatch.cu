// Bandwidth-bound kernels of the MoE layer (sm_103a): router logits for small
// E, top-k routing with the f.p statistic, the stable counting-sort dispatch,
// the weighted combine, and their backward passes; plus the router GEMMs on
// the CUDA cores for large E.
//
// Pages: "KochiLLM v1.0" model card, Architecture (shared expert + top-2 of 4
// routed, gates renormalised over the selected, E * sum f p balancing term);
// "spark-gpt" README, feature list (fp32-softmax top-k routing, statistic over
// real tokens, PAD filler positions).
#include <float.h>
#include <stdlib.h>
#include <math.h>

#include <utility>

#include "moe_common.cuh"
#include "moe_mx.cuh"
#include "moe_internal.h"

namespace moe {

namespace {

constexpr int kThreads = 256;

__device__ __forceinline__ bool row_real(const uint8_t* valid, int t) {
  return valid == nullptr || valid[t] != 0;
}

// Programmatic dependent launch: a kernel may let its successor launch while
// it still runs (griddepcontrol.launch_dependents); the successor waits for
// its predecessor's completion and memory (griddepcontrol.wait) before it
// reads the predecessor's results.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// 8 consecutive fp32 values (32-byte aligned) through the non-coherent path.
__device__ __forceinline__ void ld8f(const float* p, float* v) {
  uint4 a = ld_nc_v4(p), b = ld_nc_v4(p + 4);
  v[0] = __uint_as_float(a.x); v[1] = __uint_as_float(a.y);
  v[2] = __uint_as_float(a.z); v[3] = __uint_as_float(a.w);
  v[4] = __uint_as_float(b.x); v[5] = __uint_as_float(b.y);
  v[6] = __uint_as_float(b.z); v[7] = __uint_as_float(b.w);
}

// --------------------------------------------------------------------------
// a0 (small E): logits[t][e] = sum_c x[t][c] * Wr[c][e], one warp per token.
// Wr is staged in shared memory as [c][E] with 4 floats of padding after
// every 8 rows, so the 8 rows a lane reads sit in distinct banks.
// --------------------------------------------------------------------------
__device__ __forceinline__ int wr_smem_index(int c, int e, int E) {
  return c * E + (c >> 3) * 4 + e;
}

// Wr [d][E] fp32 -> padded shared copy, four experts of one row per 16-byte
// load (E is a multiple of 4), several loads in flight per thread.
__device__ __forceinline__ void stage_wr(const float* __restrict__ Wr, float* wr_s, int d, int E) {
  const int n4 = d * E / 4;
#pragma unroll 4
  for (int i4 = threadIdx.x; i4 < n4; i4 += blockDim.x) {
    const int i = i4 * 4, c = i / E, e = i - c * E;
    *reinterpret_cast<float4*>(wr_s + wr_smem_index(c, e, E)) =
        __ldg(reinterpret_cast<const float4*>(Wr) + i4);
  }
}

template <int E>
__global__ void __launch_bounds__(kThreads)
router_logits_small_kernel(const bf16* __restrict__ x, const float* __restrict__ Wr,
                           float* __restrict__ L, int T, int d) {
  extern __shared__ float wr_s[];
  stage_wr(Wr, wr_s, d, E);
  __syncthreads();
  const int lane = threadIdx.x & 31;
  const int wpb = blockDim.x >> 5;
  for (int t = blockIdx.x * wpb + (threadIdx.x >> 5); t < T; t += gridDim.x * wpb) {
    float acc[E];
#pragma unroll
    for (int e = 0; e < E; ++e) acc[e] = 0.f;
    const bf16* xr = x + (size_t)t * d;
    for (int c0 = lane * 8; c0 < d; c0 += 256) {
      float xf[8];
      unpack8(ld_nc_v4(xr + c0), xf);
      const float* w = wr_s + wr_smem_index(c0, 0, E);
#pragma unroll
      for (int u = 0; u < 8; ++u) {
#pragma unroll
        for (int e4 = 0; e4 < E; e4 += 4) {
          float4 wv = *reinterpret_cast<const float4*>(w + u * E + e4);
          acc[e4 + 0] = fmaf(xf[u], wv.x, acc[e4 + 0]);
          acc[e4 + 1] = fmaf(xf[u], wv.y, acc[e4 + 1]);
          acc[e4 + 2] = fmaf(xf[u], wv.z, acc[e4 + 2]);
          acc[e4 + 3] = fmaf(xf[u], wv.w, acc[e4 + 3]);
        }
      }
    }
    float mine = 0.f;
#pragma unroll
    for (int e = 0; e < E; ++e) {
      float v = warp_sum(acc[e]);
      if (lane == e) mine = v;
    }
    if (lane < E) L[(size_t)t * E + lane] = mine;
  }
}

// --------------------------------------------------------------------------
// Generic fp32 GEMM on the CUDA cores: C[m][n] = sum_k A(m,k) B(k,n).
// A(m,k) = A[m*sam + k*sak] (bf16 or fp32), B(k,n) = B[k*sbk + n*sbn] (fp32).
// 64x64 tile, 16-deep K slices, 256 threads x (4x4) outputs.  Split-K along
// gridDim.z writes partial tiles to C + z*M*N.
// --------------------------------------------------------------------------
template <typename TA>
__device__ __forceinline__ float load_as_float(const TA* p);
template <>
__device__ __forceinline__ float load_as_float<float>(const float* p) { return *p; }
template <>
__device__ __forceinline__ float load_as_float<bf16>(const bf16* p) {
  return __bfloat162float(*p);
}

template <typename TA>
__global__ void __launch_bounds__(256)
simt_gemm_kernel(const TA* __restrict__ A, long long sam, long long sak,
                 const float* __restrict__ B, long long sbk, long long sbn,
                 float* __restrict__ C, int M, int N, int K, int k_per_split) {
  __shared__ float As[16][64 + 4];
  __shared__ float Bs[16][64 + 4];
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  const int m0 = blockIdx.y * 64, n0 = blockIdx.x * 64;
  const int kbeg = blockIdx.z * k_per_split;
  const int kend = min(K, kbeg + k_per_split);
  float acc[4][4] = {};
  for (int k0 = kbeg; k0 < kend; k0 += 16) {
    for (int i = threadIdx.x; i < 16 * 64; i += 256) {
      int kk, mm;
      if (sak == 1) { mm = i / 16; kk = i % 16; } else { kk = i / 64; mm = i % 64; }
      int m = m0 + mm, k = k0 + kk;
      As[kk][mm] = (m < M && k < kend) ? load_as_float<TA>(A + m * sam + k * sak) : 0.f;
    }
    for (int i = threadIdx.x; i < 16 * 64; i += 256) {
      int kk, nn;
      if (sbn == 1) { kk = i / 64; nn = i % 64; } else { nn = i / 16; kk = i % 16; }
      int n = n0 + nn, k = k0 + kk;
      Bs[kk][nn] = (n < N && k < kend) ? B[k * sbk + n * sbn] : 0.f;
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < 16; ++kk) {
      float a[4], b[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) a[i] = As[kk][ty + 16 * i];
#pragma unroll
      for (int j = 0; j < 4; ++j) b[j] = Bs[kk][tx + 16 * j];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
    }
    __syncthreads();
  }
  float* Cz = C + (size_t)blockIdx.z * M * N;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    int m = m0 + ty + 16 * i;
    if (m >= M) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      int n = n0 + tx + 16 * j;
      if (n < N) Cz[(size_t)m * N + n] = acc[i][j];
    }
  }
}

// dW_r for small E: part[z][c][e] = sum over the tokens of slice z of
// x[t][c] * dL[t][e].  Each thread owns 8 consecutive columns (16-byte x
// loads, coalesced across the block) and walks the block's token chunk; the
// chunk's dL rows sit in shared memory.  When d/8 < blockDim.x the block's
// threads also split the chunk's tokens into `slices` interleaved sets, each
// writing its own partial.
template <int E>
__global__ void __launch_bounds__(kThreads)
router_dw_small_kernel(const bf16* __restrict__ x, const float* __restrict__ dL,
                       float* __restrict__ part, int T, int d, int tok_per_blk) {
  extern __shared__ float dl_s[];  // [tok_per_blk][E]
  const int t0 = blockIdx.x * tok_per_blk;
  const int nt = min(tok_per_blk, T - t0);
  for (int i = threadIdx.x; i < nt * E; i += blockDim.x) dl_s[i] = dL[(size_t)t0 * E + i];
  __syncthreads();
  const int groups = d / 8;
  const int slices = max(1, (int)blockDim.x / groups);
  const int s = threadIdx.x / groups;
  for (int g = threadIdx.x % groups; g < groups && s < slices; g += (slices == 1 ? blockDim.x : groups)) {
    float acc[8][E];
#pragma unroll
    for (int u = 0; u < 8; ++u)
#pragma unroll
      for (int e = 0; e < E; ++e) acc[u][e] = 0.f;
#pragma unroll 8
    for (int tl = s; tl < nt; tl += slices) {
      float xf[8];
      unpack8(ld_nc_v4(x + (size_t)(t0 + tl) * d + g * 8), xf);
      const float* dl = dl_s + tl * E;
#pragma unroll
      for (int e4 = 0; e4 < E; e4 += 4) {
        const float4 w = *reinterpret_cast<const float4*>(dl + e4);
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          acc[u][e4 + 0] = fmaf(xf[u], w.x, acc[u][e4 + 0]);
          acc[u][e4 + 1] = fmaf(xf[u], w.y, acc[u][e4 + 1]);
          acc[u][e4 + 2] = fmaf(xf[u], w.z, acc[u][e4 + 2]);
          acc[u][e4 + 3] = fmaf(xf[u], w.w, acc[u][e4 + 3]);
        }
      }
    }
    float* dst = part + ((size_t)blockIdx.x * slices + s) * d * E + (size_t)g * 8 * E;
#pragma unroll
    for (int u = 0; u < 8; ++u)
#pragma unroll
      for (int e4 = 0; e4 < E; e4 += 4)
        *reinterpret_cast<float4*>(dst + u * E + e4) =
            make_float4(acc[u][e4], acc[u][e4 + 1], acc[u][e4 + 2], acc[u][e4 + 3]);
  }
}

// Router logits on the CUDA cores for large E: L[T][E] = x[T][d] . W_r[d][E]
// with IEEE fp32 fused multiply-adds (routing decisions are taken on these
// values).  Block tile 128 tokens x BE experts x 16 of d; 256 threads, each
// owning 8 tokens x BE/16 experts; shared tiles double-buffered with the next
// slice prefetched into registers.
template <int BE>
__global__ void __launch_bounds__(256)
router_logits_sgemm_kernel(const bf16* __restrict__ x, const float* __restrict__ Wr,
                           float* __restrict__ L, int T, int d, int E, int tpb) {
  // a block computes tokens [t0, t0 + tpb) (tpb <= 128, the register tile),
  // so that the grid can be a whole number of waves over the SMs
  constexpr int BT = 128, BK = 16, TE = BE / 16;
  __shared__ __align__(16) float As[2][BK][BT + 4];
  __shared__ __align__(16) float Bs[2][BK][BE + 4];
  const int tid = threadIdx.x;
  // thread (tx, ty): tokens ty*8 .. ty*8+7 and experts 64 j + 4 tx .. +3 for
  // j < TE/4, so that each quarter-warp reads one contiguous 128-byte span of
  // the B slice (no bank conflicts)
  const int tx = tid & 15, ty = tid >> 4;
  const int t0 = blockIdx.y * tpb, e0 = blockIdx.x * BE;
  const int t_end = min(T, t0 + tpb);
  // A slice: thread -> token tid/2, k-half (tid%2)*8 (one 16-byte load)
  const int at = tid >> 1, ak = (tid & 1) * 8;
  // B slice: BK x BE floats, float4 per load
  constexpr int BV = BK * BE / 4 / 256;         // float4 loads per thread (1 or 2)
  float acc[8][TE];
#pragma unroll
  for (int i = 0; i < 8; ++i)
#pragma unroll
    for (int j = 0; j < TE; ++j) acc[i][j] = 0.f;
  uint4 areg;
  float4 breg[BV];
  auto load = [&](int k0) {
    const int t = t0 + at;
    areg = (t < t_end) ? ld_nc_v4(x + (size_t)t * d + k0 + ak) : make_uint4(0, 0, 0, 0);
#pragma unroll
    for (int v = 0; v < BV; ++v) {
      const int idx = tid + v * 256;            // float4 index in the BK x BE/4 slice
      const int kk = idx / (BE / 4), e4 = (idx % (BE / 4)) * 4;
      const int e = e0 + e4;
      breg[v] = (e < E) ? *reinterpret_cast<const float4*>(Wr + (size_t)(k0 + kk) * E + e)
                        : make_float4(0.f, 0.f, 0.f, 0.f);
    }
  };
  auto store = [&](int buf) {
    float f[8];
    unpack8(areg, f);
#pragma unroll
    for (int u = 0; u < 8; ++u) As[buf][ak + u][at] = f[u];
#pragma unroll
    for (int v = 0; v < BV; ++v) {
      const int idx = tid + v * 256;
      const int kk = idx / (BE / 4), e4 = (idx % (BE / 4)) * 4;
      *reinterpret_cast<float4*>(&Bs[buf][kk][e4]) = breg[v];
    }
  };
  load(0);
  store(0);
  __syncthreads();
  int buf = 0;
  for (int k0 = 0; k0 < d; k0 += BK) {
    const bool more = k0 + BK < d;
    if (more) load(k0 + BK);
#pragma unroll
    for (int kk = 0; kk < BK; ++kk) {
      const float4 a0 = *reinterpret_cast<const float4*>(&As[buf][kk][ty * 8]);
      const float4 a1 = *reinterpret_cast<const float4*>(&As[buf][kk][ty * 8 + 4]);
      const float a[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
      float b[TE];
#pragma unroll
      for (int j = 0; j < TE; j += 4) {
        const float4 bv = *reinterpret_cast<const float4*>(&Bs[buf][kk][(j / 4) * 64 + tx * 4]);
        b[j] = bv.x; b[j + 1] = bv.y; b[j + 2] = bv.z; b[j + 3] = bv.w;
      }
#pragma unroll
      for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < TE; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
    }
    if (more) {
      store(buf ^ 1);
      __syncthreads();
      buf ^= 1;
    }
  }
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int t = t0 + ty * 8 + i;
    if (t >= t_end) continue;
#pragma unroll
    for (int j = 0; j < TE; j += 4) {
      const int e = e0 + (j / 4) * 64 + tx * 4;
      if (e < E)
        *reinterpret_cast<float4*>(L + (size_t)t * E + e) =
            make_float4(acc[i][j], acc[i][j + 1], acc[i][j + 2], acc[i][j + 3]);
    }
  }
}

// Deterministic split reduction out[i] = sum_z part[z][i]: a block covers 32
// outputs with 8 lanes each; lane l sums z = l, l+8, ... and the 8 lane sums
// are added in lane order.
__global__ void __launch_bounds__(256)
sum_splits_kernel(const float* __restrict__ part, float* __restrict__ out, int n, int splits) {
  __shared__ float red[8][33];
  const int o = blockIdx.x * 32 + (threadIdx.x & 31);
  const int zl = threadIdx.x >> 5;
  float acc = 0.f;
  if (o < n) {
#pragma unroll 4
    for (int z = zl; z < splits; z += 8) acc += part[(size_t)z * n + o];
  }
  red[zl][threadIdx.x & 31] = acc;
  __syncthreads();
  if (zl == 0 && o < n) {
    float v = 0.f;
#pragma unroll
    for (int l = 0; l < 8; ++l) v += red[l][threadIdx.x];
    out[o] = v;
  }
}

// --------------------------------------------------------------------------
// a1: routing.  A group of G lanes (a power of two <= 32) handles one token;
// lane l of the group holds experts l, l+G, ..., (V per lane).
// --------------------------------------------------------------------------
// True if candidate (ka, ia) ranks before (kb, ib): larger key first, equal
// keys lower index first; "none" ranks last.
__device__ __forceinline__ bool ranks_before(float ka, int ia, float kb, int ib) {
  if (ia == INT_MAX) return false;
  if (ib == INT_MAX) return true;
  return ka > kb || (ka == kb && ia < ib);
}

// Routes the token held by a group of G lanes.  Lane lig of the group holds
// the logits of experts lig + G*v in lv[v] (any value where lig + G*v >= E).
// Softmax (unbiased), top-k on the biased keys with ties to the lower index,
// gates; writes topk and gates of a real token (-1 and 0 on PAD) and adds it
// to the block's counts and to this lane's statistics.
// Unsigned key that orders finite floats like the floats themselves, with
// -0 and +0 equal (both map to the key of +0); 0 is below every float's key.
__device__ __forceinline__ unsigned order_key(float x) {
  unsigned u = __float_as_uint(x);
  if (u == 0x80000000u) u = 0u;
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

template <int V>
__device__ __forceinline__ void route_token(const float (&lv_in)[V], const float* __restrict__ bias,
                                            int t, bool in_range, bool real, int E, int k, int G,
                                            int lig, int norm_topk, bool want_stats,
                                            int32_t* __restrict__ topk, float* __restrict__ gates,
                                            int* cnt_s, unsigned long long (&psum)[V],
                                            int& my_treal,
                                            float& z_acc, float& ent_acc, int* __restrict__ status) {
  float lv[V], kv[V], sv[V];
  bool bad = false;
#pragma unroll
  for (int v = 0; v < V; ++v) {
    const int e = lig + G * v;
    if (in_range && e < E) {
      lv[v] = lv_in[v];
      kv[v] = bias ? lv[v] + bias[e] : lv[v];
      bad |= !isfinite(lv[v]) || !isfinite(kv[v]);
    } else {
      lv[v] = -FLT_MAX;
      kv[v] = -FLT_MAX;
    }
  }
  if (bad && real) set_status(status, MOE_ERR_NONFINITE);
  // softmax over the E logits (unbiased)
  float m = -FLT_MAX;
#pragma unroll
  for (int v = 0; v < V; ++v) m = fmaxf(m, lv[v]);
  for (int o = G >> 1; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  float sum = 0.f;
#pragma unroll
  for (int v = 0; v < V; ++v) {
    const int e = lig + G * v;
    sv[v] = (in_range && e < E) ? expf(lv[v] - m) : 0.f;
    sum += sv[v];
  }
  for (int o = G >> 1; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
  const float rsum = 1.f / sum;
#pragma unroll
  for (int v = 0; v < V; ++v) sv[v] *= rsum;
  if (want_stats) {
    // z-loss term lse^2 and entropy lse - sum_e s_e L_e of this token
    float sl = 0.f;
#pragma unroll
    for (int v = 0; v < V; ++v)
      if (lig + G * v < E) sl = fmaf(sv[v], lv[v], sl);
    for (int o = G >> 1; o > 0; o >>= 1) sl += __shfl_xor_sync(0xffffffffu, sl, o);
    if (real && lig == 0) {
      const float lse = m + logf(sum);
      z_acc = fmaf(lse, lse, z_acc);
      ent_acc += lse - sl;
    }
  }

  // top-k
  float sel_s[V];
  int sel_i[V];
#pragma unroll
  for (int v = 0; v < V; ++v) { sel_s[v] = 0.f; sel_i[v] = -1; }
  float ssum = 0.f;
  if (G == 32) {
    // one token per warp: each lane sorts its candidates once (largest key
    // first; the sort is stable and a lane's expert indices ascend with v,
    // so equal keys keep the lower index first), then every round takes the
    // warp max of the lanes' head keys (order-preserving key bits) and the
    // lowest expert index holding it (warp min); the winning lane pops its
    // head.  k <= 32, so slot j is held by lane j.
    unsigned key[V];
    int eid[V];
    float sval[V];
#pragma unroll
    for (int v = 0; v < V; ++v) {
      const int e = lig + G * v;
      const bool ok = e < E;
      key[v] = ok ? order_key(kv[v]) : 0u;
      eid[v] = ok ? e : INT_MAX;
      sval[v] = sv[v];
    }
#pragma unroll
    for (int a = 1; a < V; ++a) {
#pragma unroll
      for (int b = a; b > 0; --b) {
        if (key[b] > key[b - 1]) {
          const unsigned tk = key[b]; key[b] = key[b - 1]; key[b - 1] = tk;
          const int te = eid[b]; eid[b] = eid[b - 1]; eid[b - 1] = te;
          const float ts = sval[b]; sval[b] = sval[b - 1]; sval[b - 1] = ts;
        }
      }
    }
    for (int j = 0; j < k; ++j) {
      const unsigned kmax = __reduce_max_sync(0xffffffffu, key[0]);
      const int win =
          __reduce_min_sync(0xffffffffu, (key[0] == kmax && kmax != 0u) ? eid[0] : INT_MAX);
      const float ws = __shfl_sync(0xffffffffu, sval[0], win == INT_MAX ? 0 : (win & 31));
      if (eid[0] == win) {
#pragma unroll
        for (int v = 0; v + 1 < V; ++v) {
          key[v] = key[v + 1]; eid[v] = eid[v + 1]; sval[v] = sval[v + 1];
        }
        key[V - 1] = 0u;
        eid[V - 1] = INT_MAX;
      }
      ssum += ws;
      if (j == lig) { sel_s[0] = ws; sel_i[0] = win; }
    }
  } else {
    // repeated group arg-max over the G lanes of the token
    unsigned taken = 0;
    for (int j = 0; j < k; ++j) {
      float bk = 0.f, bs = 0.f;
      int bi = INT_MAX;
#pragma unroll
      for (int v = 0; v < V; ++v) {
        const int e = lig + G * v;
        if (e < E && !((taken >> v) & 1u) && ranks_before(kv[v], e, bk, bi)) {
          bk = kv[v]; bi = e; bs = sv[v];
        }
      }
      for (int o = G >> 1; o > 0; o >>= 1) {
        float ok = __shfl_xor_sync(0xffffffffu, bk, o);
        int oi = __shfl_xor_sync(0xffffffffu, bi, o);
        float os = __shfl_xor_sync(0xffffffffu, bs, o);
        if (ranks_before(ok, oi, bk, bi)) { bk = ok; bi = oi; bs = os; }
      }
      // the owner of the winner marks it taken
      if (bi != INT_MAX && (bi & (G - 1)) == lig) taken |= 1u << (bi / G);
      ssum += bs;
#pragma unroll
      for (int v = 0; v < V; ++v)
        if (j == lig + G * v) { sel_s[v] = bs; sel_i[v] = bi; }
    }
  }
  if (in_range) {
#pragma unroll
    for (int v = 0; v < V; ++v) {
      const int j = lig + G * v;
      if (j < k) {
        int32_t ix = real ? sel_i[v] : -1;
        float g = real ? (norm_topk ? sel_s[v] / ssum : sel_s[v]) : 0.f;
        topk[(size_t)t * k + j] = ix;
        gates[(size_t)t * k + j] = g;
        if (real) atomicAdd(&cnt_s[sel_i[v]], 1);
      }
    }
  }
  if (real) {
    // probabilities in fixed point, 32 fractional bits, per token: integer
    // sums are exact, so p does not depend on which lane, block or kernel
    // summed which tokens
#pragma unroll
    for (int v = 0; v < V; ++v) psum[v] += __float2ull_rn(sv[v] * 4294967296.f);
    if (lig == 0) ++my_treal;
  }
}

// End of a routing block.  The block's expert counts and probability sums
// (each token's probability in fixed point with 32 fractional bits) join
// totals kept as integers by integer atomics, which are exact, so the totals
// do not depend on the order the blocks finish in, nor on how tokens were
// spread over lanes and blocks, and the last block reads only E values.
// The block's real-token count and metric sums go to per-block slots.  The
// last block to finish writes counts, f, p, aux and the metrics.
// psum_s holds [blockDim/G][E] fixed-point sums; cnt_s [E] ints with the block's counts;
// acc_cnt and acc_psum must be zero when the kernel starts.
template <int V>
__device__ __forceinline__ void route_block_end(
    const unsigned long long (&psum)[V], int my_treal, float z_acc, float ent_acc, int* cnt_s,
    unsigned long long* psum_s,
    int G, int lig, int grp, int E, int k, int* __restrict__ acc_cnt,
    unsigned long long* __restrict__ acc_psum, int* __restrict__ blk_treal,
    int* __restrict__ done, int32_t* __restrict__ counts, float* __restrict__ f,
    float* __restrict__ p, float* __restrict__ aux, float* __restrict__ blk_zent,
    float* __restrict__ stats) {
  __shared__ int treal_s, tot_s, ticket_s;
  __shared__ float red_s[32], zred_s[32], ered_s[32];        // up to 1024 threads
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int nwarps = blockDim.x >> 5;
  const int groups = blockDim.x / G;
  if (threadIdx.x == 0) { treal_s = 0; tot_s = 0; }
  __syncthreads();
#pragma unroll
  for (int v = 0; v < V; ++v) {
    const int e = lig + G * v;
    if (e < E) psum_s[grp * E + e] = psum[v];
  }
  if (lig == 0 && my_treal) atomicAdd(&treal_s, my_treal);
  if (stats) {
    z_acc = warp_sum(z_acc);
    ent_acc = warp_sum(ent_acc);
    if (lane == 0) { zred_s[warp] = z_acc; ered_s[warp] = ent_acc; }
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    unsigned long long fx = 0ull;
    for (int g2 = 0; g2 < groups; ++g2) fx += psum_s[g2 * E + e];
    if (cnt_s[e]) atomicAdd(acc_cnt + e, cnt_s[e]);
    if (fx) atomicAdd(acc_psum + e, fx);
  }
  if (threadIdx.x == 0) {
    blk_treal[blockIdx.x] = treal_s;
    if (stats) {
      float zs = 0.f, es = 0.f;
      for (int w = 0; w < nwarps; ++w) { zs += zred_s[w]; es += ered_s[w]; }
      blk_zent[2 * blockIdx.x] = zs;
      blk_zent[2 * blockIdx.x + 1] = es;
    }
  }
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) ticket_s = atomicAdd(done, 1);
  __syncthreads();
  if (ticket_s != (int)gridDim.x - 1) return;

  // last block
  __threadfence();
  const int nb = gridDim.x;
  int tr = 0;
  float zp = 0.f, ep = 0.f;
  for (int b = threadIdx.x; b < nb; b += blockDim.x) {
    tr += __ldcg(blk_treal + b);
    if (stats) {
      zp += __ldcg(blk_zent + 2 * b);
      ep += __ldcg(blk_zent + 2 * b + 1);
    }
  }
  if (tr) atomicAdd(&tot_s, tr);                 // integers: exact in any order
  if (stats) {
    zp = warp_sum(zp);
    ep = warp_sum(ep);
  }
  __syncthreads();                               // tot_s; zred_s/ered_s free again
  if (stats && lane == 0) { zred_s[warp] = zp; ered_s[warp] = ep; }
  const int Tr = tot_s;
  float part = 0.f;
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    const int c = __ldcg(acc_cnt + e);
    const double ps = (double)__ldcg(acc_psum + e) * (1.0 / 4294967296.0);
    float fe = Tr > 0 ? (float)c / (float)((long long)k * Tr) : 0.f;
    float pe = Tr > 0 ? (float)(ps / Tr) : 0.f;
    counts[e] = c;
    cnt_s[e] = c;
    f[e] = fe;
    p[e] = pe;
    part = fmaf(fe, pe, part);
  }
  part = warp_sum(part);
  if (lane == 0) red_s[warp] = part;
  __syncthreads();
  if (threadIdx.x == 0) {
    float s = 0.f;
    for (int w = 0; w < nwarps; ++w) s += red_s[w];
    aux[0] = (float)E * s;
  }
  if (stats && warp == 0) {
    // routing metrics: z-loss and entropy (warp partials in warp order), and
    // min / max / CV / unused of the counts (one warp, fixed shuffle order)
    double sum = 0.0, sq = 0.0;
    int cmin = INT_MAX, cmax = 0, unused = 0;
    for (int e = lane; e < E; e += 32) {
      const int c = cnt_s[e];
      sum += c;
      sq += (double)c * c;
      cmin = min(cmin, c);
      cmax = max(cmax, c);
      unused += c == 0;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      sum += __shfl_xor_sync(0xffffffffu, sum, o);
      sq += __shfl_xor_sync(0xffffffffu, sq, o);
      cmin = min(cmin, __shfl_xor_sync(0xffffffffu, cmin, o));
      cmax = max(cmax, __shfl_xor_sync(0xffffffffu, cmax, o));
      unused += __shfl_xor_sync(0xffffffffu, unused, o);
    }
    if (lane == 0) {
      float zs = 0.f, es = 0.f;
      for (int w = 0; w < nwarps; ++w) { zs += zred_s[w]; es += ered_s[w]; }
      const double mean = sum / E;
      const double var = fmax(sq / E - mean * mean, 0.0);
      stats[0] = Tr > 0 ? zs / (float)Tr : 0.f;
      stats[1] = Tr > 0 ? es / (float)Tr : 0.f;
      stats[2] = (float)cmin;
      stats[3] = (float)cmax;
      stats[4] = mean > 0 ? (float)(sqrt(var) / mean) : 0.f;
      stats[5] = (float)unused;
      stats[6] = (float)Tr;
      stats[7] = 0.f;
    }
  }
  if (threadIdx.x == 0) *done = 0;
}

// a1 on logits in memory.  A group of G lanes (a power of two <= 32) handles
// one token; lane l of the group holds experts l, l+G, ... (V per lane).
template <int V>
__global__ void __launch_bounds__(kThreads)
route_kernel(const float* __restrict__ L, const float* __restrict__ bias,
             const uint8_t* __restrict__ valid, int T, int E, int k, int G, int norm_topk,
             int32_t* __restrict__ topk, float* __restrict__ gates,
             int* __restrict__ acc_cnt, unsigned long long* __restrict__ acc_psum,
             int* __restrict__ blk_treal, int* __restrict__ done,
             int32_t* __restrict__ counts, float* __restrict__ f, float* __restrict__ p,
             float* __restrict__ aux, float* __restrict__ blk_zent, float* __restrict__ stats,
             int* __restrict__ status) {
  extern __shared__ unsigned char smem_raw[];
  const int groups = blockDim.x / G;
  int* cnt_s = reinterpret_cast<int*>(smem_raw);                 // [E]
  unsigned long long* psum_s = reinterpret_cast<unsigned long long*>(cnt_s + 256);  // [groups][E]
  for (int e = threadIdx.x; e < E; e += blockDim.x) cnt_s[e] = 0;
  __syncthreads();

  const int lane = threadIdx.x & 31;
  const int lig = lane & (G - 1);           // lane in group
  const int grp = threadIdx.x / G;          // group in block
  unsigned long long psum[V];
#pragma unroll
  for (int v = 0; v < V; ++v) psum[v] = 0ull;
  int my_treal = 0;
  float z_acc = 0.f, ent_acc = 0.f;

  const int tokens_per_iter = groups * gridDim.x;
  for (int t0 = blockIdx.x * groups; t0 < T; t0 += tokens_per_iter) {
    const int t = t0 + grp;
    const bool in_range = t < T;
    const bool real = in_range && row_real(valid, t);
    float lv[V];
#pragma unroll
    for (int v = 0; v < V; ++v) {
      const int e = lig + G * v;
      lv[v] = (in_range && e < E) ? L[(size_t)t * E + e] : -FLT_MAX;
    }
    route_token<V>(lv, bias, t, in_range, real, E, k, G, lig, norm_topk, stats != nullptr, topk,
                   gates, cnt_s, psum, my_treal, z_acc, ent_acc, status);
  }
  route_block_end<V>(psum, my_treal, z_acc, ent_acc, cnt_s, psum_s, G, lig, grp, E, k, acc_cnt,
                     acc_psum, blk_treal, done, counts, f, p, aux, blk_zent, stats);
}

// a0 + a1 in one pass for small E (4, 8 or 16).  A warp computes the logits
// of TT = 32/G tokens at once (G = route_group_lanes(E) = max(8, E) lanes per
// token, as in the route kernel); every W_r value read from shared memory
// serves TT tokens, and the next 256 columns of the TT rows are loaded while
// the current ones are used.  The TT*E sums are then reduced across the warp
// so that lane g*G + e ends with the logit of token g, expert e, and the
// tokens are routed in place with the route kernel's code.  The logits are
// written once (the backward reads them) and never read back.
template <int E>
__global__ void __launch_bounds__(kThreads, E < 8 ? 3 : 2)
router_route_small_kernel(const bf16* __restrict__ x, const float* __restrict__ Wr,
                          const float* __restrict__ bias, const uint8_t* __restrict__ valid,
                          int T, int d, int k, int norm_topk, float* __restrict__ L,
                          int32_t* __restrict__ topk, float* __restrict__ gates,
                          int* __restrict__ acc_cnt, unsigned long long* __restrict__ acc_psum,
                          int* __restrict__ blk_treal, int* __restrict__ done,
                          int32_t* __restrict__ counts, float* __restrict__ f,
                          float* __restrict__ p, float* __restrict__ aux,
                          float* __restrict__ blk_zent, float* __restrict__ stats,
                          int* __restrict__ status) {
  constexpr int G = E < 8 ? 8 : E;
  constexpr int TT = 32 / G;
  constexpr int N = TT * E;                      // 16 or 32 sums per warp
  extern __shared__ float wr_s[];                // padded [d][E]
  __shared__ int cnt_s[E];
  __shared__ unsigned long long psum_s[kThreads / G * E];
  stage_wr(Wr, wr_s, d, E);
  for (int e = threadIdx.x; e < E; e += blockDim.x) cnt_s[e] = 0;
  __syncthreads();
  const int lane = threadIdx.x & 31;
  const int wpb = blockDim.x >> 5;
  const int lig = lane % G, tig = lane / G;      // expert and token of this lane
  const int grp = threadIdx.x / G;
  unsigned long long psum[1] = {0ull};
  int my_treal = 0;
  float z_acc = 0.f, ent_acc = 0.f;
  for (long long tile = (long long)blockIdx.x * wpb + (threadIdx.x >> 5);
       tile * TT < T; tile += (long long)gridDim.x * wpb) {
    const int t0 = (int)(tile * TT);
    float acc[TT][E];
#pragma unroll
    for (int i = 0; i < TT; ++i)
#pragma unroll
      for (int e = 0; e < E; ++e) acc[i][e] = 0.f;
    uint4 raw[TT];
#pragma unroll
    for (int i = 0; i < TT; ++i)
      raw[i] = (t0 + i < T && lane * 8 < d) ? ld_nc_v4(x + (size_t)(t0 + i) * d + lane * 8)
                                            : make_uint4(0, 0, 0, 0);
    for (int c0 = lane * 8; c0 < d; c0 += 256) {
      uint4 cur[TT];
#pragma unroll
      for (int i = 0; i < TT; ++i) cur[i] = raw[i];
      const int cn = c0 + 256;
#pragma unroll
      for (int i = 0; i < TT; ++i)
        raw[i] = (t0 + i < T && cn < d) ? ld_nc_v4(x + (size_t)(t0 + i) * d + cn)
                                        : make_uint4(0, 0, 0, 0);
      const float* w = wr_s + wr_smem_index(c0, 0, E);
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        float xu[TT];
#pragma unroll
        for (int i = 0; i < TT; ++i) {
          const uint32_t wd = (&cur[i].x)[u >> 1];
          xu[i] = __uint_as_float((u & 1) ? (wd & 0xffff0000u) : (wd << 16));
        }
#pragma unroll
        for (int e4 = 0; e4 < E; e4 += 4) {
          const float4 wv = *reinterpret_cast<const float4*>(w + u * E + e4);
#pragma unroll
          for (int i = 0; i < TT; ++i) {
            acc[i][e4 + 0] = fmaf(xu[i], wv.x, acc[i][e4 + 0]);
            acc[i][e4 + 1] = fmaf(xu[i], wv.y, acc[i][e4 + 1]);
            acc[i][e4 + 2] = fmaf(xu[i], wv.z, acc[i][e4 + 2]);
            acc[i][e4 + 3] = fmaf(xu[i], wv.w, acc[i][e4 + 3]);
          }
        }
      }
    }
    // reduce-scatter of the N values v[j] = acc[j / E][j % E] over the warp:
    // at the step with offset o the lane keeps the half of its values that
    // its bit o selects and adds the partner's copy of that half; after
    // log2(N) steps lane l holds value l / (32 / N), summed over the lanes
    // that differ in the bits used, and the remaining offsets add the rest.
    float v[N];
#pragma unroll
    for (int j = 0; j < N; ++j) v[j] = acc[j / E][j % E];
#pragma unroll
    for (int o = 16, n = N; o > 0; o >>= 1) {
      if (n > 1) {
        const bool upper = (lane & o) != 0;
#pragma unroll
        for (int j = 0; j < n / 2; ++j) {
          const float send = upper ? v[j] : v[j + n / 2];
          const float keep = upper ? v[j + n / 2] : v[j];
          v[j] = keep + __shfl_xor_sync(0xffffffffu, send, o);
        }
        n >>= 1;
      } else {
        v[0] += __shfl_xor_sync(0xffffffffu, v[0], o);
      }
    }
    // lane l holds value j = l / (32 / N): token j / E, expert j % E.  With
    // N = 32 that is already token l / G, expert l % G; with N = 16 (E = 4,
    // G = 8) expert e of token g sits in lanes 8g + 2e and 8g + 2e + 1.
    float my = v[0];
    if (N == 16) my = __shfl_sync(0xffffffffu, my, (lane & ~7) + 2 * (lig & 3));
    const int t = t0 + tig;
    const bool in_range = t < T;
    const bool real = in_range && row_real(valid, t);
    if (in_range && lig < E) L[(size_t)t * E + lig] = my;
    float lv[1] = {my};
    route_token<1>(lv, bias, t, in_range, real, E, k, G, lig, norm_topk, stats != nullptr, topk,
                   gates, cnt_s, psum, my_treal, z_acc, ent_acc, status);
  }
  route_block_end<1>(psum, my_treal, z_acc, ent_acc, cnt_s, psum_s, G, lig, grp, E, k, acc_cnt,
                     acc_psum, blk_treal, done, counts, f, p, aux, blk_zent, stats);
}

// a0 + a1 streamed (small E, the default fused form): one resident block of
// 16 warps per SM, each block on a contiguous range of the tokens.  A warp
// works on groups of TT = 32 / G rows (or U = a multiple of TT rows when
// whole rows fit its buffers), one column chunk of CW columns at a time
// (CW = d when the rows are short).  Each warp owns two row buffers in
// shared memory: while it computes on one unit (rows x chunk), lane 0 has
// the next one in flight, loaded by untiled bulk copies (one per row, or one
// for the whole unit when it spans whole rows) that complete on the
// buffer's mbarrier, so loads need no registers and each SM keeps about 32
// units in flight.  W_r is staged meanwhile, in a layout that keeps the
// weights of two neighbouring columns side by side, so one packed fp32 FMA
// (fma.rn.f32x2) does the two columns' products for one expert: the lane
// sums even and odd columns separately and adds the two at the end.  After
// a group's last chunk its logits are reduced over the warp and the tokens
// routed with the route kernel's code.  The statistics are sums of
// integers and of per-token values, so the route kernel run on the logits
// this kernel wrote gives the same selection, gates, counts, f, p and aux.
// The kernel is launched behind the small kernel that zeroes the routing
// totals, with programmatic dependent launch: it waits for that kernel
// (griddepcontrol.wait) only before its block-end reduction.
constexpr int kStreamWarps = 16;
constexpr int kStreamThreads = kStreamWarps * 32;
constexpr int kStreamBufs = 2;                       // row buffers per warp
constexpr uint64_t kStreamWaitNs = 2000000000ull;   // a bulk copy not done in 2 s: give up

__global__ void __launch_bounds__(kThreads)
route_zero_kernel(unsigned int* __restrict__ acc, int words) {
  pdl_trigger();
  for (int i = threadIdx.x; i < words; i += blockDim.x) acc[i] = 0u;
}

// W_r [d][E] in shared memory by column pairs: every 8 columns c0..c0+7 (c0 a
// multiple of 8) take a block of 8E floats and 4 of padding (so the 8-column
// blocks of consecutive lanes fall in distinct banks); inside it, pair q
// (columns c0 + 2q and c0 + 2q + 1) holds for each expert e the two
// columns' weights side by side.
__device__ __forceinline__ int wr_pair_index(int c, int e, int E) {
  return (c >> 3) * (8 * E + 4) + ((c & 7) >> 1) * (2 * E) + 2 * e + (c & 1);
}

// Each thread moves W_r[c][e4..e4+3] and W_r[c+1][e4..e4+3] (c even) into
// the pair layout: 8 consecutive floats there.
__device__ __forceinline__ void stage_wr_pairs(const float* __restrict__ Wr, float* wr_s, int d,
                                               int E) {
  const int nq = E / 4;
  const int units = (d / 2) * nq;
#pragma unroll 4
  for (int u = threadIdx.x; u < units; u += blockDim.x) {
    const int pc = u / nq, e4 = (u - pc * nq) * 4, c = 2 * pc;
    const float4 r0 = __ldg(reinterpret_cast<const float4*>(Wr + (size_t)c * E + e4));
    const float4 r1 = __ldg(reinterpret_cast<const float4*>(Wr + (size_t)(c + 1) * E + e4));
    float* dst = wr_s + wr_pair_index(c, e4, E);
    *reinterpret_cast<float4*>(dst) = make_float4(r0.x, r1.x, r0.y, r1.y);
    *reinterpret_cast<float4*>(dst + 4) = make_float4(r0.z, r1.z, r0.w, r1.w);
  }
}

__device__ __forceinline__ unsigned long long f32x2_pack(float lo, float hi) {
  unsigned long long r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ float f32x2_sum(unsigned long long v) {
  float lo, hi;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
  return lo + hi;
}
// d = a * b + c on both halves, each an IEEE fp32 fused multiply-add.
__device__ __forceinline__ unsigned long long fma_f32x2(unsigned long long a,
                                                       unsigned long long b,
                                                       unsigned long long c) {
  unsigned long long d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}

// Warp reduce-scatter of N values, unrolled at compile time: at the step
// with offset O the lane keeps the half of its NN values that its bit O
// selects and adds the partner's copy of that half; once one value is left,
// the remaining offsets add the partners' values.  Lane l ends with value
// l / (32 / N), summed over the warp -- the same additions, in the same
// order, as the loop in router_route_small_kernel.
template <int O, int NN, int N>
struct ReduceScatter {
  static __device__ __forceinline__ void run(float (&v)[N], int lane) {
    if constexpr (NN > 1) {
      const bool upper = (lane & O) != 0;
#pragma unroll
      for (int j = 0; j < NN / 2; ++j) {
        const float send = upper ? v[j] : v[j + NN / 2];
        const float keep = upper ? v[j + NN / 2] : v[j];
        v[j] = keep + __shfl_xor_sync(0xffffffffu, send, O);
      }
      ReduceScatter<O / 2, NN / 2, N>::run(v, lane);
    } else {
      v[0] += __shfl_xor_sync(0xffffffffu, v[0], O);
      ReduceScatter<O / 2, 1, N>::run(v, lane);
    }
  }
};
template <int NN, int N>
struct ReduceScatter<0, NN, N> {
  static __device__ __forceinline__ void run(float (&)[N], int) {}
};

// One lane issues the copies of one unit -- rows [r0, r0 + rows) of x,
// columns [c0, c0 + cw) -- into a row buffer whose rows are cw_max columns
// apart, completing on the buffer's mbarrier: one copy when the unit spans
// whole rows (cw = d), else one per row.  Called after the warp has finished
// reading the buffer: the proxy fence orders those reads before the copies'
// writes.
__device__ __forceinline__ void stream_issue(const bf16* __restrict__ x, int d, int r0, int rows,
                                             int c0, int cw, int cw_max, uint32_t bar,
                                             uint32_t dst) {
  const uint32_t row_bytes = (uint32_t)cw * 2u;
  fence_proxy_async_smem();
  mbar_arrive_expect_tx(bar, (uint32_t)rows * row_bytes);
  if (cw == d) {
    bulk_load(dst, x + (size_t)r0 * d, (uint32_t)rows * row_bytes, bar);
  } else {
    for (int i = 0; i < rows; ++i)
      bulk_load(dst + (uint32_t)i * (uint32_t)cw_max * 2u, x + (size_t)(r0 + i) * d + c0,
                row_bytes, bar);
  }
}

// Unit n of a warp: row group j = n / nch (rows (ufirst + j * kStreamWarps)
// * U onwards) and column chunk n % nch; false past the block's groups.
struct StreamUnit {
  int r0, rows, ch, c0, cw;
};
__device__ __forceinline__ bool stream_unit(int n, int nch, int ufirst, int u1, int U, int T,
                                            int d, int CW, StreamUnit& s) {
  const int j = n / nch;
  const int u = ufirst + j * kStreamWarps;
  if (u >= u1) return false;
  s.ch = n - j * nch;
  s.r0 = u * U;
  s.rows = min(U, T - s.r0);
  s.c0 = s.ch * CW;
  s.cw = min(CW, d - s.c0);
  return true;
}

template <int E>
__global__ void __launch_bounds__(kStreamThreads, 1)
router_route_stream_kernel(const bf16* __restrict__ x, const float* __restrict__ Wr,
                           const float* __restrict__ bias, const uint8_t* __restrict__ valid,
                           int T, int d, int k, int norm_topk, int U, int CW, int wr_bytes,
                           int buf_bytes, float* __restrict__ L, int32_t* __restrict__ topk,
                           float* __restrict__ gates, int* __restrict__ acc_cnt,
                           unsigned long long* __restrict__ acc_psum, int* __restrict__ blk_treal,
                           int* __restrict__ done, int32_t* __restrict__ counts,
                           float* __restrict__ f, float* __restrict__ p, float* __restrict__ aux,
                           float* __restrict__ blk_zent, float* __restrict__ stats,
                           int* __restrict__ status) {
  constexpr int G = E < 8 ? 8 : E;
  constexpr int TT = 32 / G;
  constexpr int N = TT * E;                      // 16 or 32 sums per warp
  extern __shared__ __align__(128) unsigned char smem_raw[];
  float* wr_s = reinterpret_cast<float*>(smem_raw);              // column-pair layout
  unsigned char* rows_s = smem_raw + wr_bytes;                   // [warps][bufs][buf_bytes]
  __shared__ __align__(8) uint64_t full[kStreamWarps * kStreamBufs];
  __shared__ int cnt_s[E];
  __shared__ unsigned long long psum_s[kStreamThreads / G * E];
  __shared__ int abort_s;                        // stays 0: waits end only by time

  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int lig = lane % G, tig = lane / G;      // expert and token of this lane
  const int grp = threadIdx.x / G;
  const int nch = (d + CW - 1) / CW;             // > 1 only with U == TT
  const int ngroups = (T + U - 1) / U;
  const int per = (ngroups + gridDim.x - 1) / gridDim.x;
  const int u0 = blockIdx.x * per;
  const int u1 = min(ngroups, u0 + per);
  const int ufirst = u0 + warp;
  if (threadIdx.x < kStreamWarps * kStreamBufs) mbar_init(smem_u32(&full[threadIdx.x]), 1);
  if (threadIdx.x == 0) abort_s = 0;
  for (int e = threadIdx.x; e < E; e += blockDim.x) cnt_s[e] = 0;
  fence_mbar_init();
  __syncthreads();

  const uint32_t bar0 = smem_u32(&full[warp * kStreamBufs]);
  const uint32_t dst0 = smem_u32(rows_s + (size_t)warp * kStreamBufs * buf_bytes);
  if (lane == 0) {
    StreamUnit su;
#pragma unroll
    for (int n = 0; n < kStreamBufs; ++n)
      if (stream_unit(n, nch, ufirst, u1, U, T, d, CW, su))
        stream_issue(x, d, su.r0, su.rows, su.c0, su.cw, CW, bar0 + 8 * n, dst0 + n * buf_bytes);
  }
  stage_wr_pairs(Wr, wr_s, d, E);
  __syncthreads();

  unsigned long long psum[1] = {0ull};
  int my_treal = 0;
  float z_acc = 0.f, ent_acc = 0.f;
  unsigned long long acc2[TT][E];                // (even, odd) column sums of one group
  StreamUnit su;
  for (int n = 0; stream_unit(n, nch, ufirst, u1, U, T, d, CW, su); ++n) {
    const int b = n % kStreamBufs;
    // each warp waits only for its own copies (never on another warp)
    if (!mbar_wait_bounded(bar0 + 8 * b, (uint32_t)((n / kStreamBufs) & 1), &abort_s,
                           kStreamWaitNs)) {
      if (lane == 0) set_status(status, MOE_ERR_TIMEOUT);
      // wait (bounded) for this warp's other copy in flight, so that none
      // still targets the buffers when the block exits
      StreamUnit sn;
      if (stream_unit(n + 1, nch, ufirst, u1, U, T, d, CW, sn))
        mbar_wait_bounded(bar0 + 8 * ((n + 1) % kStreamBufs),
                          (uint32_t)(((n + 1) / kStreamBufs) & 1), &abort_s, kStreamWaitNs);
      break;
    }
    const bf16* xs = reinterpret_cast<const bf16*>(
        rows_s + ((size_t)warp * kStreamBufs + b) * buf_bytes);
    for (int g0 = 0; g0 < su.rows; g0 += TT) {
      if (su.ch == 0) {
#pragma unroll
        for (int i = 0; i < TT; ++i)
#pragma unroll
          for (int e = 0; e < E; ++e) acc2[i][e] = 0ull;
      }
      for (int cc = lane * 8; cc < su.cw; cc += 256) {
        uint4 cur[TT];
#pragma unroll
        for (int i = 0; i < TT; ++i)
          cur[i] = g0 + i < su.rows
                       ? *reinterpret_cast<const uint4*>(xs + (size_t)(g0 + i) * CW + cc)
                       : make_uint4(0, 0, 0, 0);
        const float* w = wr_s + wr_pair_index(su.c0 + cc, 0, E);
#pragma unroll
        for (int q = 0; q < 4; ++q) {            // columns +2q, +2q+1
          unsigned long long xp[TT];
#pragma unroll
          for (int i = 0; i < TT; ++i) {
            const uint32_t wd = (&cur[i].x)[q];
            xp[i] = f32x2_pack(__uint_as_float(wd << 16), __uint_as_float(wd & 0xffff0000u));
          }
#pragma unroll
          for (int e2 = 0; e2 < E; e2 += 2) {
            const float4 wv = *reinterpret_cast<const float4*>(w + q * 2 * E + 2 * e2);
            const unsigned long long wa = f32x2_pack(wv.x, wv.y);
            const unsigned long long wb = f32x2_pack(wv.z, wv.w);
#pragma unroll
            for (int i = 0; i < TT; ++i) {
              acc2[i][e2] = fma_f32x2(xp[i], wa, acc2[i][e2]);
              acc2[i][e2 + 1] = fma_f32x2(xp[i], wb, acc2[i][e2 + 1]);
            }
          }
        }
      }
      if (su.ch == nch - 1) {
        float v[N];
#pragma unroll
        for (int jj = 0; jj < N; ++jj) v[jj] = f32x2_sum(acc2[jj / E][jj % E]);
        ReduceScatter<16, N, N>::run(v, lane);
        // lane l holds value l / (32 / N): token (l / (32 / N)) / E; with
        // N = 16 (E = 4, G = 8) expert e of token g sits in lanes 8g + 2e, +1
        float my = v[0];
        if (N == 16) my = __shfl_sync(0xffffffffu, my, (lane & ~7) + 2 * (lig & 3));
        const int t = su.r0 + g0 + tig;
        const bool in_range = g0 + tig < su.rows;
        const bool real = in_range && row_real(valid, t);
        if (in_range && lig < E) L[(size_t)t * E + lig] = my;
        float lv[1] = {my};
        route_token<1>(lv, bias, t, in_range, real, E, k, G, lig, norm_topk, stats != nullptr,
                       topk, gates, cnt_s, psum, my_treal, z_acc, ent_acc, status);
      }
    }
    __syncwarp();
    if (lane == 0) {
      StreamUnit sn;
      if (stream_unit(n + kStreamBufs, nch, ufirst, u1, U, T, d, CW, sn))
        stream_issue(x, d, sn.r0, sn.rows, sn.c0, sn.cw, CW, bar0 + 8 * b, dst0 + b * buf_bytes);
    }
  }
  pdl_wait();                                    // the zeroed totals
  route_block_end<1>(psum, my_treal, z_acc, ent_acc, cnt_s, psum_s, G, lig, grp, E, k, acc_cnt,
                     acc_psum, blk_treal, done, counts, f, p, aux, blk_zent, stats);
}

// --------------------------------------------------------------------------
// Data-parallel routing statistics: a rank's sums, and f / p / aux from sums
// that the caller has added over the ranks.  One block; E <= 256.
// --------------------------------------------------------------------------
__global__ void __launch_bounds__(kThreads)
route_partials_kernel(const int32_t* __restrict__ counts, const float* __restrict__ p, int E,
                      int k, double* __restrict__ sums) {
  __shared__ long long tot_s;
  if (threadIdx.x == 0) {
    long long m = 0;
    for (int e = 0; e < E; ++e) m += counts[e];
    tot_s = m;
  }
  __syncthreads();
  const double Tr = (double)(tot_s / k);
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    sums[e] = (double)counts[e];
    sums[E + e] = (double)p[e] * Tr;
  }
  if (threadIdx.x == 0) sums[2 * E] = Tr;
}

__global__ void __launch_bounds__(kThreads)
route_finalize_kernel(const double* __restrict__ sums, int E, int k, float* __restrict__ f,
                      float* __restrict__ p, float* __restrict__ aux) {
  __shared__ double red[kThreads];
  const double T = sums[2 * E];
  double part = 0.0;
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    const double fe = T > 0 ? sums[e] / ((double)k * T) : 0.0;
    const double pe = T > 0 ? sums[E + e] / T : 0.0;
    f[e] = (float)fe;
    p[e] = (float)pe;
    part += fe * pe;
  }
  red[threadIdx.x] = part;
  __syncthreads();
  if (threadIdx.x == 0) {
    double s = 0.0;
    for (int i = 0; i < (int)blockDim.x; ++i) s += red[i];
    aux[0] = (float)((double)E * s);
  }
}

// --------------------------------------------------------------------------
// a2: stable counting-sort dispatch.  Its three kernels run back to back with
// programmatic dependent launch: the histogram and the scan let their
// successor launch while they still run (griddepcontrol.launch_dependents),
// and the scan and the scatter wait for their predecessor's completion and
// memory (griddepcontrol.wait) before they read its results, so the launch
// latency of the two small kernels overlaps the work.
// --------------------------------------------------------------------------

__global__ void __launch_bounds__(kThreads)
perm_hist_kernel(const int32_t* __restrict__ topk, int T, int k, int E,
                 int* __restrict__ hist, int* __restrict__ status) {
  pdl_trigger();
  __shared__ int h[256];
  for (int e = threadIdx.x; e < E; e += blockDim.x) h[e] = 0;
  __syncthreads();
  const long long q0 = (long long)blockIdx.x * kPermChunk * k;
  const long long q1 = min((long long)T * k, q0 + (long long)kPermChunk * k);
  for (long long q = q0 + threadIdx.x; q < q1; q += blockDim.x) {
    int e = topk[q];
    if (e >= E) set_status(status, MOE_ERR_INDEX);
    else if (e >= 0) atomicAdd(&h[e], 1);
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) hist[(size_t)blockIdx.x * E + e] = h[e];
}

// Counts, offsets, padded row offsets and, for every (block, expert), the
// first row that block writes for that expert.  Each expert's blocks are split
// into contiguous ranges over kScanThreads / E threads: range sums, an
// exclusive prefix over the ranges, then each thread walks its own range.
constexpr int kScanThreads = 1024;
__global__ void __launch_bounds__(kScanThreads)
perm_scan_kernel(const int* __restrict__ hist, int nblk, int E, int32_t* __restrict__ counts,
                 int32_t* __restrict__ offsets, int32_t* __restrict__ row_offsets,
                 int* __restrict__ base) {
  pdl_wait();
  pdl_trigger();
  __shared__ int part[kScanThreads];
  __shared__ int cnt_s[257];
  __shared__ int off_s[257];
  __shared__ int roff_s[257];
  const int G = blockDim.x / E;                  // ranges per expert (E <= 256)
  const int e = threadIdx.x % E, g = threadIdx.x / E;
  const bool act = g < G;
  const int b0 = act ? (int)((long long)g * nblk / G) : 0;
  const int b1 = act ? (int)((long long)(g + 1) * nblk / G) : 0;
  int local = 0;
#pragma unroll 4
  for (int b = b0; b < b1; ++b) local += hist[(size_t)b * E + e];
  if (act) part[g * E + e] = local;
  __syncthreads();
  int pre = 0;
  if (act) {
    for (int g2 = 0; g2 < g; ++g2) pre += part[g2 * E + e];
    if (g == G - 1) cnt_s[e] = pre + local;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    int o = 0, ro = 0;
    for (int x = 0; x < E; ++x) {
      off_s[x] = o;
      roff_s[x] = ro;
      o += cnt_s[x];
      ro += (cnt_s[x] + kRowAlign - 1) / kRowAlign * kRowAlign;
    }
    off_s[E] = o;
    roff_s[E] = ro;
  }
  __syncthreads();
  for (int x = threadIdx.x; x <= E; x += blockDim.x) {
    offsets[x] = off_s[x];
    row_offsets[x] = roff_s[x];
    if (x < E) counts[x] = cnt_s[x];
  }
  if (act) {
    int run = roff_s[e] + pre;
    for (int b = b0; b < b1; ++b) {
      base[(size_t)b * E + e] = run;
      run += hist[(size_t)b * E + e];
    }
  }
}

// Ranks each (t, j) pair of the block's token chunk in pair order with one
// warp (warp match + popc per 32 pairs, on the chunk's expert ids staged in
// shared memory by one coalesced load), then copies each token's x row once
// into its k destination rows, several 16-byte vectors in flight per lane.
// The block also zeroes the pad rows of the experts e = blockIdx.x (mod
// gridDim.x).  MX: instead of bf16 rows it writes each token's row quantised
// to MXFP8 (e4m3 codes [R][d] and the UE8M0 scale atoms of x_s, blocks of 32
// along d), quantising the row once for its k destinations.
constexpr int kScatterThreads = 512;
template <bool MX>
__global__ void __launch_bounds__(kScatterThreads, 2)
perm_scatter_kernel(const bf16* __restrict__ x, const int32_t* __restrict__ topk, int T,
                    int d, int k, int E, const int* __restrict__ base,
                    const int32_t* __restrict__ counts, const int32_t* __restrict__ row_offsets,
                    int32_t* __restrict__ perm, int32_t* __restrict__ inv,
                    bf16* __restrict__ x_perm, uint8_t* __restrict__ x_q,
                    uint8_t* __restrict__ x_s, uint8_t* __restrict__ xt_q,
                    uint8_t* __restrict__ xt_s, int Tp) {
  pdl_wait();
  __shared__ int base_s[256];
  __shared__ int dest_s[kPermChunk * kMaxK];     // expert ids, then destination rows
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int t_beg = blockIdx.x * kPermChunk;
  const int t_end = min(T, t_beg + kPermChunk);
  const int npairs = (t_end - t_beg) * k;
  for (int e = threadIdx.x; e < E; e += blockDim.x) base_s[e] = base[(size_t)blockIdx.x * E + e];
  for (int ql = threadIdx.x; ql < npairs; ql += blockDim.x)
    dest_s[ql] = topk[(size_t)t_beg * k + ql];
  __syncthreads();
  if (warp == 0) {
    const unsigned lt = (1u << lane) - 1u;
    for (int q0 = 0; q0 < npairs; q0 += 32) {
      const int ql = q0 + lane;
      const int e = ql < npairs ? dest_s[ql] : -1;
      const bool ok = e >= 0 && e < E;
      const unsigned act = __ballot_sync(0xffffffffu, ok);
      int dest = -1;
      unsigned peers = 0;
      if (ok) {
        peers = __match_any_sync(act, e);
        dest = base_s[e] + __popc(peers & lt);
      }
      __syncwarp();
      if (ok && lane == 31 - __clz(peers)) base_s[e] += __popc(peers);
      if (ql < npairs) dest_s[ql] = dest;
      __syncwarp();
    }
  }
  __syncthreads();
  for (int ql = threadIdx.x; ql < npairs; ql += blockDim.x) {
    const int dest = dest_s[ql];
    const long long q = (long long)t_beg * k + ql;
    inv[q] = dest;
    if (dest >= 0) perm[dest] = (int32_t)q;
  }
  // row copies: one warp per token, each x row read once (skipped when the
  // gate/up GEMM gathers its rows from x itself: x_perm == NULL)
  constexpr int U = 4;                           // 16-byte vectors in flight per lane
  const int wpb = blockDim.x >> 5;
  const int nb32 = d / 32, kg = d / 128;          // MX: blocks per row, atoms per row block
  // MX: 8 consecutive values per lane as in the bf16 copy (d a multiple of
  // 256, so every lane runs the same column loop), each block of 32 shared
  // by four lanes whose maximum comes from shuffles (mx_quant8x4)
  for (int tl = warp; MX && tl < t_end - t_beg; tl += wpb) {
    const bf16* src = x + (size_t)(t_beg + tl) * d;
    const int* dst = dest_s + tl * k;
    const int t = t_beg + tl;
    const bool real = dst[0] >= 0;
    for (int c00 = 0; c00 < d; c00 += 256 * U) {
      uint4 raw[U];
      uint32_t q[U][2], sb[U];
#pragma unroll
      for (int u = 0; u < U; ++u)
        if (c00 + u * 256 < d) raw[u] = ld_nc_v4(src + c00 + u * 256 + lane * 8);
#pragma unroll
      for (int u = 0; u < U; ++u) {
        if (c00 + u * 256 >= d) break;               // uniform over the warp
        float v[8];
        unpack8(raw[u], v);
        sb[u] = mx_quant8x4(v, q[u]);
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int c0 = c00 + u * 256 + lane * 8;
        if (c00 + u * 256 >= d) break;
        const int b = c0 >> 5;
        if (xt_q != nullptr) {
          // the same codes in token order for the shared expert; PAD tokens
          // (no destination row) as zeros
          *reinterpret_cast<uint2*>(xt_q + (size_t)t * d + c0) =
              real ? make_uint2(q[u][0], q[u][1]) : make_uint2(0, 0);
          if ((lane & 3) == 0)
            xt_s[((size_t)(t >> 7) * kg + (b >> 2)) * kMxAtom + mx_sf_byte(t & 127, b & 3)] =
                real ? (uint8_t)sb[u] : (uint8_t)0;
        }
        for (int j = 0; j < k; ++j) {
          const int r = dst[j];
          if (r < 0) continue;
          *reinterpret_cast<uint2*>(x_q + (size_t)r * d + c0) = make_uint2(q[u][0], q[u][1]);
          if ((lane & 3) == 0)
            x_s[((size_t)(r >> 7) * kg + (b >> 2)) * kMxAtom + mx_sf_byte(r & 127, b & 3)] =
                (uint8_t)sb[u];
          // training: the bf16 rows too (weight gradients)
          if (x_perm != nullptr) st_v4(x_perm + (size_t)r * d + c0, raw[u]);
        }
      }
    }
  }
  for (int tl = warp; !MX && x_perm != nullptr && tl < t_end - t_beg; tl += wpb) {
    const bf16* src = x + (size_t)(t_beg + tl) * d;
    const int* dst = dest_s + tl * k;
    for (int c0 = lane * 8; c0 < d; c0 += 256 * U) {
      uint4 v[U];
#pragma unroll
      for (int u = 0; u < U; ++u)
        if (c0 + u * 256 < d) v[u] = ld_nc_v4(src + c0 + u * 256);
      for (int j = 0; j < k; ++j) {
        const int r = dst[j];
        if (r < 0) continue;
        bf16* o = x_perm + (size_t)r * d + c0;
#pragma unroll
        for (int u = 0; u < U; ++u)
          if (c0 + u * 256 < d) st_v4(o + u * 256, v[u]);
      }
    }
  }
  // the token-order copy's padding rows [T, Tp) as zeros (the last block)
  if (MX && xt_q != nullptr && blockIdx.x == gridDim.x - 1) {
    for (int r = T + warp; r < Tp; r += wpb) {
      for (int c0 = lane * 16; c0 < d; c0 += 512)
        st_v4(xt_q + (size_t)r * d + c0, make_uint4(0, 0, 0, 0));
      for (int b = lane; b < nb32; b += 32)
        xt_s[((size_t)(r >> 7) * kg + (b >> 2)) * kMxAtom + mx_sf_byte(r & 127, b & 3)] = 0;
    }
  }
  // zero pad rows
  for (int e = blockIdx.x; e < E; e += gridDim.x) {
    const int r0 = row_offsets[e] + counts[e];
    const int r1 = row_offsets[e + 1];
    for (int r = r0 + warp; r < r1; r += wpb) {
      if (lane == 0) perm[r] = -1;
      if (x_perm != nullptr)
        for (int c0 = lane * 8; c0 < d; c0 += 256)
          st_v4(x_perm + (size_t)r * d + c0, make_uint4(0, 0, 0, 0));
      if (MX) {
        for (int c0 = lane * 16; c0 < d; c0 += 512)
          st_v4(x_q + (size_t)r * d + c0, make_uint4(0, 0, 0, 0));
        for (int b = lane; b < nb32; b += 32)
          x_s[((size_t)(r >> 7) * kg + (b >> 2)) * kMxAtom + mx_sf_byte(r & 127, b & 3)] = 0;
      }
    }
  }
}

// --------------------------------------------------------------------------
// a6: y[t] = sum_j g[t][j] out_perm[inv[t][j]] (+ s_out[t]); one warp/token.
// --------------------------------------------------------------------------
__global__ void __launch_bounds__(kThreads)
combine_kernel(const bf16* __restrict__ out_perm, const int32_t* __restrict__ inv,
               const float* __restrict__ gates, const uint8_t* __restrict__ valid,
               const float* __restrict__ s_out, bf16* __restrict__ y, int T, int d, int k,
               long long rows, int* status) {
  const int lane = threadIdx.x & 31;
  const int wpb = blockDim.x >> 5;
  for (int t = blockIdx.x * wpb + (threadIdx.x >> 5); t < T; t += gridDim.x * wpb) {
    const bool real = row_real(valid, t);
    int my_r = -1;
    float my_g = 0.f;
    if (lane < k && real) {
      my_r = dbg_row(inv[(size_t)t * k + lane], rows, status);
      my_g = gates[(size_t)t * k + lane];
    }
    bf16* yr = y + (size_t)t * d;
    for (int c0 = lane * 8; c0 < d; c0 += 256) {
      float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
      if (real) {
        for (int j = 0; j < k; ++j) {
          const int r = __shfl_sync(0xffffffffu, my_r, j);
          const float g = __shfl_sync(0xffffffffu, my_g, j);
          if (r < 0) continue;
          float v[8];
          unpack8(ld_nc_v4(out_perm + (size_t)r * d + c0), v);
#pragma unroll
          for (int u = 0; u < 8; ++u) acc[u] = fmaf(g, v[u], acc[u]);
        }
        if (s_out) {
          float v[8];
          ld8f(s_out + (size_t)t * d + c0, v);
#pragma unroll
          for (int u = 0; u < 8; ++u) acc[u] += v[u];
        }
      }
      st_v4(yr + c0, pack8(acc));
    }
  }
}

// --------------------------------------------------------------------------
// a7 (i) + (vii): combine backward and the router-logit gradient.
// d_out[inv[t,j]] = g[t,j] dY[t];  dg[t,j] = <dY[t], out_perm[inv[t,j]]>;
// d_logits from dg through the gate map, plus the aux term
// (aux_coef E / T_real) s_e (f_e - sum_i f_i s_i).  Also zeroes d_out pad rows.
// With dq (the MXFP8 training step; d a multiple of 256, so every lane runs
// the same column loop), the fp32 g dY is also quantised along d into e4m3
// codes dq [R][d] and scale atoms ds [R/128][d/128], pad rows as zeros.
// --------------------------------------------------------------------------
template <int V>
__global__ void __launch_bounds__(kThreads)
combine_bwd_kernel(const bf16* __restrict__ dY, const bf16* __restrict__ out_perm,
                   const int32_t* __restrict__ inv, const int32_t* __restrict__ topk,
                   const float* __restrict__ gates, const float* __restrict__ L,
                   const float* __restrict__ f, const int32_t* __restrict__ counts,
                   const uint8_t* __restrict__ valid, const int32_t* __restrict__ row_offsets,
                   bf16* __restrict__ d_out, uint8_t* __restrict__ dq,
                   uint8_t* __restrict__ ds, float* __restrict__ d_logits, int T, int d, int E,
                   int k, int norm_topk, float aux_coef, float z_coef, long long rows,
                   int* status) {
  __shared__ float f_s[256];
  __shared__ float coef_s, zcoef_s;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int wpb = blockDim.x >> 5;
  for (int e = threadIdx.x; e < E; e += blockDim.x) f_s[e] = f[e];
  if (threadIdx.x == 0) {
    long long m = 0;
    for (int e = 0; e < E; ++e) m += counts[e];
    const long long Tr = m / k;
    coef_s = Tr > 0 ? aux_coef * (float)E / (float)Tr : 0.f;
    zcoef_s = Tr > 0 ? 2.f * z_coef / (float)Tr : 0.f;
  }
  __syncthreads();
  const float coef = coef_s;
  const float zcoef = zcoef_s;
  for (int t = blockIdx.x * wpb + warp; t < T; t += gridDim.x * wpb) {
    const bool real = row_real(valid, t);
    float* dl = d_logits + (size_t)t * E;
    if (!real) {
      for (int e = lane; e < E; e += 32) dl[e] = 0.f;
      continue;
    }
    int my_r = -1, my_i = -1;
    float my_g = 0.f;
    if (lane < k) {
      my_r = dbg_row(inv[(size_t)t * k + lane], rows, status);
      my_i = topk[(size_t)t * k + lane];
      my_g = gates[(size_t)t * k + lane];
    }
    const bf16* dyr = dY + (size_t)t * d;
    float my_dg = 0.f;
    for (int j = 0; j < k; ++j) {
      const int r = __shfl_sync(0xffffffffu, my_r, j);
      const float g = __shfl_sync(0xffffffffu, my_g, j);
      float dot = 0.f;
      if (r >= 0) {
        for (int c0 = lane * 8; c0 < d; c0 += 256) {
          float dy[8], o[8], go[8];
          unpack8(ld_nc_v4(dyr + c0), dy);
          unpack8(ld_nc_v4(out_perm + (size_t)r * d + c0), o);
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            dot = fmaf(dy[u], o[u], dot);
            go[u] = g * dy[u];
          }
          st_v4(d_out + (size_t)r * d + c0, pack8(go));
          if (dq != nullptr) {
            uint32_t cq[2];
            const uint32_t sb = mx_quant8x4(go, cq);
            *reinterpret_cast<uint2*>(dq + (size_t)r * d + c0) = make_uint2(cq[0], cq[1]);
            if ((lane & 3) == 0)
              ds[((size_t)(r >> 7) * (d >> 7) + (c0 >> 7)) * kMxAtom +
                 mx_sf_byte(r & 127, (c0 >> 5) & 3)] = (uint8_t)sb;
          }
        }
      }
      dot = warp_sum(dot);
      if (lane == j) my_dg = dot;
    }
    // sum_j g_j dg_j (slot order)
    float gdg = 0.f;
    for (int j = 0; j < k; ++j)
      gdg = fmaf(__shfl_sync(0xffffffffu, my_g, j), __shfl_sync(0xffffffffu, my_dg, j), gdg);
    // softmax of the logits (for the aux term and the no-renorm map)
    float lv[V], sv[V];
    float m = -FLT_MAX;
#pragma unroll
    for (int v = 0; v < V; ++v) {
      const int e = lane + 32 * v;
      lv[v] = e < E ? L[(size_t)t * E + e] : -FLT_MAX;
      m = fmaxf(m, lv[v]);
    }
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    float sum = 0.f;
#pragma unroll
    for (int v = 0; v < V; ++v) {
      const int e = lane + 32 * v;
      sv[v] = e < E ? expf(lv[v] - m) : 0.f;
      sum += sv[v];
    }
    sum = warp_sum(sum);
    const float lse = m + logf(sum);
    float fs = 0.f;
#pragma unroll
    for (int v = 0; v < V; ++v) {
      const int e = lane + 32 * v;
      sv[v] = sv[v] / sum;
      if (e < E) fs = fmaf(f_s[e], sv[v], fs);
    }
    fs = warp_sum(fs);
    float main[V];
#pragma unroll
    for (int v = 0; v < V; ++v) main[v] = 0.f;
    for (int j = 0; j < k; ++j) {
      const int ej = __shfl_sync(0xffffffffu, my_i, j);
      const float dgj = __shfl_sync(0xffffffffu, my_dg, j);
      const float gj = __shfl_sync(0xffffffffu, my_g, j);
#pragma unroll
      for (int v = 0; v < V; ++v)
        if (lane + 32 * v == ej) main[v] += norm_topk ? gj * (dgj - gdg) : sv[v] * dgj;
    }
#pragma unroll
    for (int v = 0; v < V; ++v) {
      const int e = lane + 32 * v;
      if (e >= E) continue;
      float mv = main[v];
      if (!norm_topk) mv -= sv[v] * gdg;
      // aux term with f held constant, and the z-loss term 2 z lse s / T_real
      dl[e] = mv + coef * sv[v] * (f_s[e] - fs) + zcoef * lse * sv[v];
    }
  }
  // zero d_out pad rows
  for (int e = blockIdx.x; e < E; e += gridDim.x) {
    const int r0 = row_offsets[e] + counts[e];
    const int r1 = row_offsets[e + 1];
    for (int r = r0 + warp; r < r1; r += wpb)
      for (int c0 = lane * 8; c0 < d; c0 += 256) {
        st_v4(d_out + (size_t)r * d + c0, make_uint4(0, 0, 0, 0));
        if (dq != nullptr) {
          *reinterpret_cast<uint2*>(dq + (size_t)r * d + c0) = make_uint2(0, 0);
          if ((lane & 3) == 0)
            ds[((size_t)(r >> 7) * (d >> 7) + (c0 >> 7)) * kMxAtom +
               mx_sf_byte(r & 127, (c0 >> 5) & 3)] = 0;
        }
      }
  }
}

// --------------------------------------------------------------------------
// a7 (vi), layers without a shared expert: dx[t] = sum_j dx_perm[inv[t,j]]
// + d_logits[t] Wr^T (with a shared expert the same sum runs in the shared
// expert's dx GEMM epilogue).  The router term comes from dxr (large E) or
// from Wr staged in shared memory (small E).  PAD rows get 0.
// --------------------------------------------------------------------------
template <int ES>
__global__ void __launch_bounds__(kThreads)
dx_gather_kernel(const bf16* __restrict__ dx_perm, const int32_t* __restrict__ inv,
                 const float* __restrict__ dxr,
                 const float* __restrict__ dL, const float* __restrict__ Wr,
                 const uint8_t* __restrict__ valid, bf16* __restrict__ dx, int T, int d,
                 int k, long long rows, int* status) {
  extern __shared__ float wr_s[];
  if constexpr (ES > 0) {
    for (int i = threadIdx.x; i < d * ES; i += blockDim.x) {
      int c = i / ES, e = i - c * ES;
      wr_s[wr_smem_index(c, e, ES)] = Wr[i];
    }
    __syncthreads();
  }
  const int lane = threadIdx.x & 31;
  const int wpb = blockDim.x >> 5;
  for (int t = blockIdx.x * wpb + (threadIdx.x >> 5); t < T; t += gridDim.x * wpb) {
    const bool real = row_real(valid, t);
    int my_r = -1;
    if (lane < k && real) my_r = dbg_row(inv[(size_t)t * k + lane], rows, status);
    float dl[ES > 0 ? ES : 1];
    if constexpr (ES > 0) {
#pragma unroll
      for (int e = 0; e < ES; ++e) dl[e] = real ? dL[(size_t)t * ES + e] : 0.f;
    }
    for (int c0 = lane * 8; c0 < d; c0 += 256) {
      float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
      if (real) {
        for (int j = 0; j < k; ++j) {
          const int r = __shfl_sync(0xffffffffu, my_r, j);
          if (r < 0) continue;
          float v[8];
          unpack8(ld_nc_v4(dx_perm + (size_t)r * d + c0), v);
#pragma unroll
          for (int u = 0; u < 8; ++u) acc[u] += v[u];
        }
        if constexpr (ES > 0) {
          const float* w = wr_s + wr_smem_index(c0, 0, ES);
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            float s = 0.f;
#pragma unroll
            for (int e4 = 0; e4 < ES; e4 += 4) {
              float4 wv = *reinterpret_cast<const float4*>(w + u * ES + e4);
              s = fmaf(dl[e4 + 0], wv.x, s);
              s = fmaf(dl[e4 + 1], wv.y, s);
              s = fmaf(dl[e4 + 2], wv.z, s);
              s = fmaf(dl[e4 + 3], wv.w, s);
            }
            acc[u] += s;
          }
        } else if (dxr) {
          const float4* pr = reinterpret_cast<const float4*>(dxr + (size_t)t * d + c0);
          float4 a = pr[0], b = pr[1];
          acc[0] += a.x; acc[1] += a.y; acc[2] += a.z; acc[3] += a.w;
          acc[4] += b.x; acc[5] += b.y; acc[6] += b.z; acc[7] += b.w;
        }
      }
      st_v4(dx + (size_t)t * d + c0, pack8(acc));
    }
  }
}

int grid_for(int items_per_block, long long items, int cap) {
  long long g = (items + items_per_block - 1) / items_per_block;
  if (g < 1) g = 1;
  if (g > cap) g = cap;
  return (int)g;
}

int small_E(int E) { return (E == 4 || E == 8 || E == 16) ? E : 0; }

// --------------------------------------------------------------------------
// Self-test of the GEMM kernels' failure path on a wait that cannot complete: one thread
// waits, with the same bounded wait, on an mbarrier that nothing arrives on;
// after `limit_ns` it gives up and latches MOE_ERR_TIMEOUT in the status word,
// as the GEMM roles do, and the kernel returns normally.
__global__ void wait_timeout_selftest_kernel(int* status, unsigned long long limit_ns) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    if (!mbar_wait_bounded(smem_u32(&bar), 0, &abort_flag, limit_ns))
      set_status(status, MOE_ERR_TIMEOUT);
  }
}

}  // namespace

int route_group_lanes(int E) {
  int G = 8;
  while (G < E && G < 32) G <<= 1;
  return G;
}

bool router_small_path(const moe_config& c) {
  const int es = small_E(c.E);
  return es > 0 && (size_t)c.d * es * 4 + (size_t)(c.d / 8) * 16 <= 96 * 1024;
}

static size_t wr_smem_bytes(int d, int E) { return (size_t)d * E * 4 + (size_t)(d / 8 + 1) * 16; }

cudaError_t launch_router_logits(const moe_config& c, const void* x, const float* Wr, float* L,
                                 cudaStream_t s) {
  DeviceInfo di;
  if (device_info(&di) != MOE_OK) return cudaErrorUnknown;
  if (router_small_path(c)) {
    const size_t smem = wr_smem_bytes(c.d, c.E);
    const int grid = grid_for(kThreads / 32, c.T, di.num_sms * 4);
    const bf16* xb = static_cast<const bf16*>(x);
    switch (c.E) {
      case 4:
        cudaFuncSetAttribute(router_logits_small_kernel<4>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        router_logits_small_kernel<4><<<grid, kThreads, smem, s>>>(xb, Wr, L, c.T, c.d);
        break;
      case 8:
        cudaFuncSetAttribute(router_logits_small_kernel<8>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        router_logits_small_kernel<8><<<grid, kThreads, smem, s>>>(xb, Wr, L, c.T, c.d);
        break;
      default:
        cudaFuncSetAttribute(router_logits_small_kernel<16>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        router_logits_small_kernel<16><<<grid, kThreads, smem, s>>>(xb, Wr, L, c.T, c.d);
        break;
    }
    return cudaGetLastError();
  }
  if (c.E % 32 == 0 && c.d % 16 == 0) {
    // L[T][E] = x[T][d] . Wr[d][E], register-tiled fp32 FMA
    // token blocks: ceil(T / 128) rounded up to whole waves (SMs x resident
    // blocks per SM for the expert columns of one block row), each block
    // taking ceil(T / blocks) <= 128 tokens; a token's arithmetic does not
    // depend on its block
    DeviceInfo di;
    if (device_info(&di) != MOE_OK) return cudaErrorUnknown;
    auto waves = [&](auto kern, int gx) {
      int per_sm = 0;
      if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, 256, 0) != cudaSuccess ||
          per_sm < 1) {
        cudaGetLastError();
        per_sm = 1;
      }
      const long long slots = (long long)di.num_sms * per_sm;
      long long by = (c.T + 127) / 128;
      const long long total = by * gx;
      if (total % slots != 0 && total > slots / 2) {
        const long long want = (total + slots - 1) / slots * slots;
        by = (want + gx - 1) / gx;
      }
      const int tpb = (int)((c.T + by - 1) / by);
      return std::make_pair(dim3((unsigned)gx, (unsigned)((c.T + tpb - 1) / tpb), 1), tpb);
    };
    if (c.E % 128 == 0) {
      const auto g = waves(router_logits_sgemm_kernel<128>, c.E / 128);
      router_logits_sgemm_kernel<128><<<g.first, 256, 0, s>>>(static_cast<const bf16*>(x), Wr,
                                                              L, c.T, c.d, c.E, g.second);
    } else {
      const auto g = waves(router_logits_sgemm_kernel<64>, (c.E + 63) / 64);
      router_logits_sgemm_kernel<64><<<g.first, 256, 0, s>>>(static_cast<const bf16*>(x), Wr,
                                                             L, c.T, c.d, c.E, g.second);
    }
    return cudaGetLastError();
  }
  // L[T][E] = x[T][d] . Wr[d][E]
  dim3 grid((c.E + 63) / 64, (c.T + 63) / 64, 1);
  simt_gemm_kernel<bf16><<<grid, 256, 0, s>>>(static_cast<const bf16*>(x), c.d, 1, Wr, c.E, 1,
                                               L, c.T, c.E, c.d, c.d);
  return cudaGetLastError();
}

cudaError_t launch_router_dx(const moe_config& c, const float* dL, const float* Wr, float* dxr,
                             cudaStream_t s) {
  // dxr[T][d] = dL[T][E] . Wr^T ; B(k=e, n=c) = Wr[c*E + e]
  dim3 grid((c.d + 63) / 64, (c.T + 63) / 64, 1);
  simt_gemm_kernel<float><<<grid, 256, 0, s>>>(dL, c.E, 1, Wr, 1, c.E, dxr, c.T, c.d, c.E, c.E);
  return cudaGetLastError();
}

// Small-E dW_r: tokens per block.  128 tokens per slice, so the partial
// count (blocks x slices, summed afterwards) stays near T / 128 whatever d is.
int router_dw_small_chunk(const moe_config& c) {
  const int groups = c.d / 8;
  const int slices = groups >= kThreads ? 1 : kThreads / groups;
  // the block's dL rows (chunk x E fp32) stay within 48 KB of shared memory
  const int cap = (48 * 1024 / (4 * c.E)) / kDwTokPerBlk * kDwTokPerBlk;
  const int chunk = kDwTokPerBlk * slices;
  return chunk < cap ? chunk : cap;
}

int router_dw_small_parts(const moe_config& c) {
  const int groups = c.d / 8;
  const int slices = groups >= kThreads ? 1 : kThreads / groups;
  const int chunk = router_dw_small_chunk(c);
  return (c.T + chunk - 1) / chunk * slices;
}

cudaError_t launch_router_dw(const moe_config& c, const void* x, const float* dL, float* dWr,
                             float* part, int splits, cudaStream_t s) {
  if (router_small_path(c)) {
    const int chunk = router_dw_small_chunk(c);
    const int nblk = (c.T + chunk - 1) / chunk;
    const int nparts = router_dw_small_parts(c);
    const size_t smem = (size_t)chunk * c.E * sizeof(float);
    const bf16* xb = static_cast<const bf16*>(x);
    // exactly groups x slices threads (no idle thread when d/8 < 256)
    const int groups = c.d / 8;
    const int threads = groups >= kThreads ? kThreads : groups * (kThreads / groups);
    switch (c.E) {
      case 4:
        router_dw_small_kernel<4><<<nblk, threads, smem, s>>>(xb, dL, part, c.T, c.d, chunk);
        break;
      case 8:
        router_dw_small_kernel<8><<<nblk, threads, smem, s>>>(xb, dL, part, c.T, c.d, chunk);
        break;
      default:
        router_dw_small_kernel<16><<<nblk, threads, smem, s>>>(xb, dL, part, c.T, c.d, chunk);
        break;
    }
    const int n = c.d * c.E;
    sum_splits_kernel<<<(n + 31) / 32, 256, 0, s>>>(part, dWr, n, nparts);
    return cudaGetLastError();
  }
  // dWr[d][E] = sum_t x[t][c] dL[t][e]: A(m=c, k=t) = x[t*d + c]
  const int kps = ((c.T + splits - 1) / splits + 15) / 16 * 16;
  dim3 grid((c.E + 63) / 64, (c.d + 63) / 64, splits);
  simt_gemm_kernel<bf16><<<grid, 256, 0, s>>>(static_cast<const bf16*>(x), 1, c.d, dL, c.E, 1,
                                               part, c.d, c.E, c.T, kps);
  const int n = c.d * c.E;
  sum_splits_kernel<<<(n + 31) / 32, 256, 0, s>>>(part, dWr, n, splits);
  return cudaGetLastError();
}

cudaError_t launch_sum_splits(const float* part, float* out, int n, int splits, cudaStream_t s) {
  sum_splits_kernel<<<(n + 31) / 32, 256, 0, s>>>(part, out, n, splits);
  return cudaGetLastError();
}

cudaError_t launch_route(const moe_config& c, const float* L, const float* bias,
                         const uint8_t* valid, int32_t* topk, float* gates, int32_t* counts,
                         float* f, float* p, float* aux, float* stats, char* ws,
                         const WsLayout& w, cudaStream_t s) {
  const int G = route_group_lanes(c.E);
  const int V = (c.E + G - 1) / G;
  const int groups = kThreads / G;
  const size_t smem = 256 * sizeof(int) + (size_t)groups * c.E * sizeof(unsigned long long);
  char* acc = ws + w.route_done;
  cudaError_t err = cudaMemsetAsync(acc, 0, kRouteAccBytes, s);
  if (err != cudaSuccess) return err;
  int* done = reinterpret_cast<int*>(acc);
  int* cnt = reinterpret_cast<int*>(acc + kRouteAccCnt);
  unsigned long long* psum = reinterpret_cast<unsigned long long*>(acc + kRouteAccPsum);
  int* treal = reinterpret_cast<int*>(ws + w.route_treal);
  float* zent = reinterpret_cast<float*>(ws + w.route_zent);
  int* status = reinterpret_cast<int*>(ws + w.status);
  const int grid = w.route_blocks;
#define MOE_ROUTE(VV)                                                                        \
  cudaFuncSetAttribute(route_kernel<VV>, cudaFuncAttributeMaxDynamicSharedMemorySize,        \
                       (int)smem);                                                           \
  route_kernel<VV><<<grid, kThreads, smem, s>>>(L, bias, valid, c.T, c.E, c.k, G, c.norm_topk, \
                                                topk, gates, cnt, psum, treal, done, counts, f, \
                                                p, aux, zent, stats, status)
  if (V <= 1) { MOE_ROUTE(1); }
  else if (V <= 2) { MOE_ROUTE(2); }
  else if (V <= 4) { MOE_ROUTE(4); }
  else { MOE_ROUTE(8); }
#undef MOE_ROUTE
  return cudaGetLastError();
}

// The route kernel with caller-chosen scratch pointers and grid size (used by
// the entry point whose scratch is a fixed device array instead of a
// workspace).  Same kernel, same arithmetic.
cudaError_t launch_route_scratch(const moe_config& c, const float* L, const float* bias,
                                 const uint8_t* valid, int32_t* topk, float* gates,
                                 int32_t* counts, float* f, float* p, float* aux, char* acc,
                                 int* blk_treal, int* status, int grid, cudaStream_t s) {
  const int G = route_group_lanes(c.E);
  const int V = (c.E + G - 1) / G;
  const int groups = kThreads / G;
  const size_t smem = 256 * sizeof(int) + (size_t)groups * c.E * sizeof(unsigned long long);
  cudaError_t err = cudaMemsetAsync(acc, 0, kRouteAccBytes, s);
  if (err != cudaSuccess) return err;
  int* done = reinterpret_cast<int*>(acc);
  int* acc_cnt = reinterpret_cast<int*>(acc + kRouteAccCnt);
  unsigned long long* acc_psum = reinterpret_cast<unsigned long long*>(acc + kRouteAccPsum);
#define MOE_ROUTE_S(VV)                                                                       \
  cudaFuncSetAttribute(route_kernel<VV>, cudaFuncAttributeMaxDynamicSharedMemorySize,         \
                       (int)smem);                                                            \
  route_kernel<VV><<<grid, kThreads, smem, s>>>(L, bias, valid, c.T, c.E, c.k, G, c.norm_topk, \
                                                topk, gates, acc_cnt, acc_psum, blk_treal, done, \
                                                counts, f, p, aux, nullptr, nullptr, status)
  if (V <= 1) { MOE_ROUTE_S(1); }
  else if (V <= 2) { MOE_ROUTE_S(2); }
  else if (V <= 4) { MOE_ROUTE_S(4); }
  else { MOE_ROUTE_S(8); }
#undef MOE_ROUTE_S
  return cudaGetLastError();
}

// A kernel launch with dynamic shared memory that may begin while the
// previous kernel on the stream still runs (programmatic stream
// serialisation); the kernel calls griddepcontrol.wait before it reads what
// that kernel wrote.
template <typename... K, typename... A>
cudaError_t launch_pdl_smem(void (*kern)(K...), dim3 grid, dim3 block, size_t smem,
                            cudaStream_t s, A... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, kern, args...);
  return e != cudaSuccess ? e : cudaGetLastError();
}

// Units and buffers of router_route_stream_kernel: two buffers per warp,
// each at most 1/32 of what W_r leaves of the 227 KB a block may use.  When
// TT whole rows fit a buffer, a unit is U = TT * m whole rows (CW = d);
// otherwise it is TT rows by a chunk of CW columns (a multiple of 256).
// False if not even TT rows of 256 columns fit.
bool router_stream_sizes(const moe_config& c, int* U, int* CW, int* wr_bytes, int* buf_bytes) {
  const int G = route_group_lanes(c.E);
  const int TT = 32 / G;
  const int wr = (int)((wr_smem_bytes(c.d, c.E) + 127) / 128 * 128);
  // static shared memory: mbarriers, counts, per-group sums, block-end scratch
  const int static_smem = 1024 + (kStreamThreads / G) * c.E * 8 + 512;
  int per_buf = (227 * 1024 - wr - static_smem) / (kStreamWarps * kStreamBufs);
  if (per_buf > 8 * 1024) per_buf = 8 * 1024;
  const int row_bytes = c.d * 2;
  if (TT * row_bytes <= per_buf) {
    *U = TT * (per_buf / (TT * row_bytes));
    *CW = c.d;
  } else {
    const int cw = per_buf / (TT * 2) / 256 * 256;
    if (cw < 256) return false;
    *U = TT;
    *CW = cw;
  }
  *wr_bytes = wr;
  *buf_bytes = (*U * *CW * 2 + 127) / 128 * 128;
  return true;
}

cudaError_t launch_router_route(const moe_config& c, const void* x, const float* Wr,
                                const float* bias, const uint8_t* valid, float* L, int32_t* topk,
                                float* gates, int32_t* counts, float* f, float* p, float* aux,
                                float* stats, char* ws, const WsLayout& w, cudaStream_t s) {
  int U = 0, CW = 0, wrb = 0, bufb = 0;
  DeviceInfo di;
  if (device_info(&di) != MOE_OK) return cudaErrorUnknown;
  // MOE_ROUTER_STREAM=0 selects the register-loading form (comparisons)
  const char* env = getenv("MOE_ROUTER_STREAM");
  const bool stream_form = !(env && env[0] == '0');
  if (stream_form && router_stream_sizes(c, &U, &CW, &wrb, &bufb)) {
    char* acc = ws + w.route_done;
    route_zero_kernel<<<1, kThreads, 0, s>>>(reinterpret_cast<unsigned int*>(acc),
                                             (int)(kRouteAccBytes / 4));
    cudaError_t err = cudaGetLastError();
    if (err != cudaSuccess) return err;
    int* done = reinterpret_cast<int*>(acc);
    int* cnt = reinterpret_cast<int*>(acc + kRouteAccCnt);
    unsigned long long* psum = reinterpret_cast<unsigned long long*>(acc + kRouteAccPsum);
    int* treal = reinterpret_cast<int*>(ws + w.route_treal);
    float* zent = reinterpret_cast<float*>(ws + w.route_zent);
    int* status = reinterpret_cast<int*>(ws + w.status);
    const long long ngroups = ((long long)c.T + U - 1) / U;
    long long grid = di.num_sms;
    if (grid > ngroups) grid = ngroups;
    if (grid > w.route_blocks) grid = w.route_blocks;   // its per-block slots
    if (grid < 1) grid = 1;
    const size_t smem = (size_t)wrb + (size_t)kStreamWarps * kStreamBufs * bufb;
    const bf16* xb = static_cast<const bf16*>(x);
#define MOE_RRS(EE)                                                                           \
  cudaFuncSetAttribute(router_route_stream_kernel<EE>,                                        \
                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);               \
  return launch_pdl_smem(router_route_stream_kernel<EE>, dim3((unsigned)grid),                \
                         dim3(kStreamThreads), smem, s, xb, Wr, bias, valid, c.T, c.d, c.k,   \
                         c.norm_topk, U, CW, wrb, bufb, L, topk, gates, cnt, psum, treal,     \
                         done, counts, f, p, aux, zent, stats, status)
    if (c.E == 4) { MOE_RRS(4); }
    else if (c.E == 8) { MOE_RRS(8); }
    else { MOE_RRS(16); }
#undef MOE_RRS
  }
  const size_t smem = wr_smem_bytes(c.d, c.E);
  char* acc = ws + w.route_done;
  cudaError_t err = cudaMemsetAsync(acc, 0, kRouteAccBytes, s);
  if (err != cudaSuccess) return err;
  int* done = reinterpret_cast<int*>(acc);
  int* cnt = reinterpret_cast<int*>(acc + kRouteAccCnt);
  unsigned long long* psum = reinterpret_cast<unsigned long long*>(acc + kRouteAccPsum);
  int* treal = reinterpret_cast<int*>(ws + w.route_treal);
  float* zent = reinterpret_cast<float*>(ws + w.route_zent);
  int* status = reinterpret_cast<int*>(ws + w.status);
  const int grid = w.route_blocks;        // 256 / E tokens per block and pass, as for route
  const bf16* xb = static_cast<const bf16*>(x);
#define MOE_RR(EE)                                                                            \
  cudaFuncSetAttribute(router_route_small_kernel<EE>,                                         \
                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);               \
  router_route_small_kernel<EE><<<grid, kThreads, smem, s>>>(                                 \
      xb, Wr, bias, valid, c.T, c.d, c.k, c.norm_topk, L, topk, gates, cnt, psum, treal, done, \
      counts, f, p, aux, zent, stats, status)
  if (c.E == 4) { MOE_RR(4); }
  else if (c.E == 8) { MOE_RR(8); }
  else { MOE_RR(16); }
#undef MOE_RR
  return cudaGetLastError();
}

cudaError_t launch_wait_timeout_selftest(int* status, unsigned long long limit_ns,
                                         cudaStream_t s) {
  wait_timeout_selftest_kernel<<<1, 32, 0, s>>>(status, limit_ns);
  return cudaGetLastError();
}

cudaError_t launch_route_partials(const moe_config& c, const int32_t* counts, const float* p,
                                  double* sums, cudaStream_t s) {
  route_partials_kernel<<<1, kThreads, 0, s>>>(counts, p, c.E, c.k, sums);
  return cudaGetLastError();
}

cudaError_t launch_route_finalize(const moe_config& c, const double* sums, float* f, float* p,
                                  float* aux, cudaStream_t s) {
  route_finalize_kernel<<<1, kThreads, 0, s>>>(sums, c.E, c.k, f, p, aux);
  return cudaGetLastError();
}

// A launch that may begin while the previous kernel on the stream still runs
// (programmatic stream serialisation); the kernel waits for that kernel's
// completion with griddepcontrol.wait before it reads the kernel's results.
template <typename... K, typename... A>
cudaError_t launch_pdl(void (*kern)(K...), dim3 grid, dim3 block, cudaStream_t s, A... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = 0;
  cfg.stream = s;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, kern, args...);
  return e != cudaSuccess ? e : cudaGetLastError();
}

cudaError_t launch_permute(const moe_config& c, const void* x, const int32_t* topk,
                           int32_t* counts, int32_t* offsets, int32_t* row_offsets,
                           int32_t* perm, int32_t* inv, void* x_perm, char* ws,
                           const WsLayout& w, cudaStream_t s) {
  int* hist = reinterpret_cast<int*>(ws + w.perm_hist);
  int* base = reinterpret_cast<int*>(ws + w.perm_base);
  int* status = reinterpret_cast<int*>(ws + w.status);
  const int nblk = w.perm_blocks;
  perm_hist_kernel<<<nblk, kThreads, 0, s>>>(topk, c.T, c.k, c.E, hist, status);
  launch_pdl(perm_scan_kernel, dim3(1), dim3(kScanThreads), s, (const int*)hist, nblk, c.E,
             counts, offsets, row_offsets, base);
  return launch_pdl(perm_scatter_kernel<false>, dim3(nblk), dim3(kScatterThreads), s,
                    static_cast<const bf16*>(x), topk, c.T, c.d, c.k, c.E, (const int*)base,
                    (const int32_t*)counts, (const int32_t*)row_offsets, perm, inv,
                    static_cast<bf16*>(x_perm), (uint8_t*)nullptr, (uint8_t*)nullptr,
                    (uint8_t*)nullptr, (uint8_t*)nullptr, 0);
}

cudaError_t launch_permute_mx(const moe_config& c, const void* x, const int32_t* topk,
                              int32_t* counts, int32_t* offsets, int32_t* row_offsets,
                              int32_t* perm, int32_t* inv, uint8_t* x_q, uint8_t* x_s,
                              uint8_t* xt_q, uint8_t* xt_s, void* x_perm, char* ws,
                              const WsLayout& w, cudaStream_t s) {
  int* hist = reinterpret_cast<int*>(ws + w.perm_hist);
  int* base = reinterpret_cast<int*>(ws + w.perm_base);
  int* status = reinterpret_cast<int*>(ws + w.status);
  const int nblk = w.perm_blocks;
  perm_hist_kernel<<<nblk, kThreads, 0, s>>>(topk, c.T, c.k, c.E, hist, status);
  launch_pdl(perm_scan_kernel, dim3(1), dim3(kScanThreads), s, (const int*)hist, nblk, c.E,
             counts, offsets, row_offsets, base);
  return launch_pdl(perm_scatter_kernel<true>, dim3(nblk), dim3(kScatterThreads), s,
                    static_cast<const bf16*>(x), topk, c.T, c.d, c.k, c.E, (const int*)base,
                    (const int32_t*)counts, (const int32_t*)row_offsets, perm, inv,
                    static_cast<bf16*>(x_perm), x_q, x_s, xt_q, xt_s, (c.T + 127) / 128 * 128);
}

cudaError_t launch_combine(const moe_config& c, const void* out_perm, const int32_t* inv,
                           const float* gates, const uint8_t* valid, const float* s_out,
                           void* y, long long rows, int* status, cudaStream_t s) {
  DeviceInfo di;
  if (device_info(&di) != MOE_OK) return cudaErrorUnknown;
  const int grid = grid_for(kThreads / 32, c.T, di.num_sms * 8);
  combine_kernel<<<grid, kThreads, 0, s>>>(static_cast<const bf16*>(out_perm), inv, gates,
                                           valid, s_out,
                                           static_cast<bf16*>(y), c.T, c.d, c.k, rows, status);
  return cudaGetLastError();
}

cudaError_t launch_combine_bwd(const moe_config& c, const void* dY, const void* out_perm,
                               const int32_t* inv, const int32_t* topk, const float* gates,
                               const float* L, const float* f, const int32_t* counts,
                               const uint8_t* valid, const int32_t* row_offsets, void* d_out,
                               uint8_t* dout_q, uint8_t* dout_s, float* d_logits, long long rows,
                               int* status, cudaStream_t s) {
  if (dout_q != nullptr && (c.d % 256 != 0 || dout_s == nullptr)) return cudaErrorInvalidValue;
  DeviceInfo di;
  if (device_info(&di) != MOE_OK) return cudaErrorUnknown;
  const int grid = grid_for(kThreads / 32, c.T, di.num_sms * 8);
  const int V = (c.E + 31) / 32;
#define MOE_CBWD(VV)                                                                          \
  combine_bwd_kernel<VV><<<grid, kThreads, 0, s>>>(                                           \
      static_cast<const bf16*>(dY), static_cast<const bf16*>(out_perm), inv, topk, gates, L, f, \
      counts, valid, row_offsets, static_cast<bf16*>(d_out), dout_q, dout_s, d_logits, c.T,    \
      c.d, c.E, c.k,                                                                           \
      c.norm_topk, c.aux_coef, c.z_coef, rows, status)
  if (V <= 1) { MOE_CBWD(1); }
  else if (V <= 2) { MOE_CBWD(2); }
  else if (V <= 4) { MOE_CBWD(4); }
  else { MOE_CBWD(8); }
#undef MOE_CBWD
  return cudaGetLastError();
}

cudaError_t launch_dx_gather(const moe_config& c, const void* dx_perm, const int32_t* inv,
                             const float* dxr, const float* d_logits,
                             const float* Wr, const uint8_t* valid, void* dx, long long rows,
                             int* status, cudaStream_t s) {
  DeviceInfo di;
  if (device_info(&di) != MOE_OK) return cudaErrorUnknown;
  const int grid = grid_for(kThreads / 32, c.T, di.num_sms * 4);
  const bf16* dp = static_cast<const bf16*>(dx_perm);
  bf16* o = static_cast<bf16*>(dx);
  if (router_small_path(c)) {
    const size_t smem = wr_smem_bytes(c.d, c.E);
#define MOE_DXG(EE)                                                                           \
  cudaFuncSetAttribute(dx_gather_kernel<EE>, cudaFuncAttributeMaxDynamicSharedMemorySize,     \
                       (int)smem);                                                            \
  dx_gather_kernel<EE><<<grid, kThreads, smem, s>>>(dp, inv, nullptr, d_logits, Wr, valid, o, \
                                                    c.T, c.d, c.k, rows, status)
    if (c.E == 4) { MOE_DXG(4); }
    else if (c.E == 8) { MOE_DXG(8); }
    else { MOE_DXG(16); }
#undef MOE_DXG
  } else {
    dx_gather_kernel<0><<<grid, kThreads, 0, s>>>(dp, inv, dxr, d_logits, Wr, valid, o, c.T,
                                                  c.d, c.k, rows, status);
  }
  return cudaGetLastError();
}

}  // namespace moe
