// MXFP8 routed experts on the 5th-generation tensor cores (sm_103a).
//
// "KohakUwULLM" README, Key features and Selected measurements: MXFP8 (e4m3
// values, UE8M0 scales per 32 values) on the routed experts, with fully fused
// expert kernels that never materialise the (tokens * top_k, hidden)
// intermediates in 16-bit form.
//
// Here that is:
//   * a weight quantiser (bf16 W_gu, W_down -> e4m3 codes + scale atoms);
//   * the quantising permute (moe_dispatch.cu, perm_scatter_kernel<true>);
//   * a persistent grouped GEMM on tcgen05.mma kind::mxf8f6f4 with block
//     scales: TMA brings 128 x 128-byte tiles of codes (128-byte swizzle) and
//     a bulk copy brings each stage's two 512-byte scale atoms; the MMA thread
//     moves the atoms into TMEM with tcgen05.cp and issues four K = 32 MMAs
//     per stage, each picking its K-block's scale byte by the scale-factor id;
//   * epilogues: gate/up -> h = silu(a) * b quantised straight to MXFP8 (codes
//     and scale atoms of h, no bf16 h); down -> out_perm fp32 for the combine.
// One CTA per SM, 128 x 128 tiles, double-buffered 128-column accumulators;
// the scale slots of the six stages take TMEM columns 256-303.
#include <algorithm>
#include <cstring>
#include <mutex>

#include "moe_common.cuh"
#include "moe_internal.h"
#include "moe_mx.cuh"

namespace moe {

namespace {

constexpr int XBM = 128;                    // tile rows
constexpr int XBN = 128;                    // tile columns (UMMA N)
constexpr int XBK = 128;                    // K per stage: one 128-byte row of e4m3
constexpr int XUK = 32;                     // K per MMA (= one scale block)
constexpr int XA_BYTES = XBM * XBK;         // 16 KB
constexpr int XB_BYTES = XBN * XBK;         // 16 KB
constexpr int XSTAGE = XA_BYTES + XB_BYTES;
constexpr int XSTAGES = 6;
constexpr int XSF_BYTES = 2 * kMxAtom;      // per stage: the A atom, then the B atom
constexpr int XTHREADS = 384;               // warp 0 TMA, 1 MMA, 2 TMEM, 4-11 epilogue
constexpr int XEPI0 = 4;
constexpr int XEPI_THREADS = 256;
constexpr int XTMEM_COLS = 512;
constexpr int XSF_COL = 2 * XBN;            // stage s scales: columns 256 + 8 s (A), + 4 (B)
constexpr uint64_t XWAIT_NS = 2000000000ull;  // bounded waits give up after 2 s
constexpr uint64_t XDRAIN_NS = 200000000ull;
constexpr size_t XRESERVE = 2048;           // struct XShared
constexpr size_t XSMEM = XRESERVE + 1024 + (size_t)XSTAGES * (XSTAGE + XSF_BYTES);
static_assert(XSMEM <= 232448, "exceeds the 227 KB opt-in shared memory of a block");
static_assert(XSF_COL + 8 * XSTAGES <= XTMEM_COLS, "scale slots exceed the TMEM allocation");

enum MxKind { MXK_GATE_UP = 0, MXK_DOWN = 1 };

struct XParams {
  const int32_t* row_offsets;  // [E+1] padded segment offsets (multiples of 128)
  int E;
  int K;                       // reduction length (multiple of 128)
  int H;                       // hidden size (gate/up: output units; down: K)
  int d;                       // model dim
  int n_tiles;                 // column tiles per 128-row block
  int kg;                      // K / 128: scale atoms per row block
  int nbt;                     // weight scale blocks per expert
  const uint8_t* sfa;          // activation scale atoms [R/128][kg][512]
  const uint8_t* sfb;          // weight scale atoms [E][nbt][kg][512]
  uint8_t* hq;                 // gate/up: h codes [R][H]
  uint8_t* hs;                 // gate/up: h scale atoms [R/128][H/128][512]
  float* out;                  // down: out_perm [R][d] fp32
  int* status;
};

struct XShared {
  uint64_t full[XSTAGES];
  uint64_t empty[XSTAGES];
  uint64_t tfull[2];
  uint64_t tempty[2];
  uint64_t drain;
  uint32_t tmem_base;
  int abort_flag;
  int roff[257];
};
static_assert(sizeof(XShared) <= XRESERVE, "bookkeeping too large");

struct XTile {
  int e, m0, n0;
};

// Last index i in [0, n) with a[i] <= v (a non-decreasing, a[0] <= v).
__device__ __forceinline__ int x_last_le(const int* a, int n, int v) {
  int lo = 0, hi = n - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (a[mid] <= v) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// Tile idx: 128-row block idx / n_tiles of the padded permuted rows, column
// tile idx % n_tiles (64 hidden units = 64 gate + 64 up weight rows for
// gate/up, 128 model columns for down).
template <int KIND>
__device__ __forceinline__ XTile x_tile(const XParams& p, const XShared& sh, int idx) {
  XTile t;
  const int mu = idx / p.n_tiles;
  t.n0 = (idx - mu * p.n_tiles) * (KIND == MXK_GATE_UP ? XBN / 2 : XBN);
  t.m0 = mu * XBM;
  t.e = x_last_le(sh.roff, p.E, t.m0);
  return t;
}

__device__ __forceinline__ void x_fail(XShared& sh, int* status) {
  set_status(status, MOE_ERR_TIMEOUT);
  *(volatile int*)&sh.abort_flag = 1;
}

// The logistic function with CUDA's fast exponential and approximate
// division; the result is quantised to e4m3 (3 mantissa bits) right after.
__device__ __forceinline__ float x_silu(float a) { return __fdividef(a, 1.f + __expf(-a)); }


// ------------------------------------------------------------------ kernel
template <int KIND>
__global__ void __launch_bounds__(XTHREADS, 1)
mx_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
               const XParams p) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t ring = (raw + (uint32_t)XRESERVE + 1023u) & ~1023u;
  const uint32_t sfring = ring + (uint32_t)(XSTAGES * XSTAGE);
  if (sfring + (uint32_t)(XSTAGES * XSF_BYTES) - raw > (uint32_t)XSMEM) {
    if (threadIdx.x == 0) set_status(p.status, MOE_ERR_DEVICE);
    return;
  }
  XShared& sh = *reinterpret_cast<XShared*>(smem_raw);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < XSTAGES; ++s) {
      mbar_init(smem_u32(&sh.full[s]), 1);
      mbar_init(smem_u32(&sh.empty[s]), 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(smem_u32(&sh.tfull[a]), 1);
      mbar_init(smem_u32(&sh.tempty[a]), XEPI_THREADS);
    }
    mbar_init(smem_u32(&sh.drain), 1);
    sh.abort_flag = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
  }
  for (int e = threadIdx.x; e <= p.E; e += blockDim.x) sh.roff[e] = p.row_offsets[e];
  if (warp == 2) {
    tmem_alloc(smem_u32(&sh.tmem_base), XTMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sh.tmem_base;
  volatile int* abort_flag = &sh.abort_flag;
  const int ntiles = (sh.roff[p.E] / XBM) * p.n_tiles;

  if (warp == 0 && lane == 0) {
    // ---------------- producer: codes by TMA, scale atoms by bulk copy
    int stage = 0;
    uint32_t phase = 0;
    int pending[XSTAGES];
    for (int s = 0; s < XSTAGES; ++s) pending[s] = -1;
    bool ok = true;
    for (int idx = blockIdx.x; idx < ntiles && ok; idx += gridDim.x) {
      const XTile t = x_tile<KIND>(p, sh, idx);
      const int jb = KIND == MXK_GATE_UP ? t.n0 / (XBN / 2) : t.n0 / XBN;
      const uint8_t* sfa = p.sfa + (size_t)(t.m0 / XBM) * p.kg * kMxAtom;
      const uint8_t* sfb = p.sfb + ((size_t)t.e * p.nbt + jb) * p.kg * kMxAtom;
      for (int kb = 0; kb < p.kg; ++kb) {
        if (!mbar_wait_bounded(smem_u32(&sh.empty[stage]), phase ^ 1u, abort_flag, XWAIT_NS)) {
          x_fail(sh, p.status);
          ok = false;
          break;
        }
        const uint32_t fb = smem_u32(&sh.full[stage]);
        const uint32_t sa = ring + stage * XSTAGE;
        const uint32_t sb = sa + XA_BYTES;
        const uint32_t sf = sfring + stage * XSF_BYTES;
        mbar_arrive_expect_tx(fb, XSTAGE + XSF_BYTES);
        tma_load_2d(sa, &tmA, fb, kb * XBK, t.m0);
        if (KIND == MXK_GATE_UP) {
          // 64 gate rows then the 64 up rows of the same hidden units
          tma_load_4d(sb, &tmB, fb, kb * XBK, t.n0, 0, t.e);
          tma_load_4d(sb + XB_BYTES / 2, &tmB, fb, kb * XBK, t.n0, 1, t.e);
        } else {
          tma_load_3d(sb, &tmB, fb, kb * XBK, t.n0, t.e);
        }
        bulk_load(sf, sfa + (size_t)kb * kMxAtom, kMxAtom, fb);
        bulk_load(sf + kMxAtom, sfb + (size_t)kb * kMxAtom, kMxAtom, fb);
        pending[stage] = (int)phase;
        if (++stage == XSTAGES) { stage = 0; phase ^= 1u; }
      }
    }
    if (!ok) {
      // let every copy already issued land before shared memory is released
      for (int s = 0; s < XSTAGES; ++s)
        if (pending[s] >= 0) {
          int dummy = 0;
          mbar_wait_bounded(smem_u32(&sh.full[s]), (uint32_t)pending[s], &dummy, XDRAIN_NS);
        }
    }
  } else if (warp == 1 && lane == 0) {
    // ---------------- MMA issuer
    constexpr uint32_t idesc0 = umma_idesc_mx(XBM, XBN);
    int stage = 0;
    uint32_t phase = 0;
    int it = 0;
    bool ok = true;
    for (int idx = blockIdx.x; idx < ntiles && ok; idx += gridDim.x, ++it) {
      const int acc = it & 1;
      const uint32_t acc_phase = (it >> 1) & 1;
      if (!mbar_wait_bounded(smem_u32(&sh.tempty[acc]), acc_phase ^ 1u, abort_flag, XWAIT_NS)) {
        x_fail(sh, p.status);
        break;
      }
      tc_fence_after();
      const uint32_t d_tmem = tmem + acc * XBN;
      for (int kb = 0; kb < p.kg; ++kb) {
        if (!mbar_wait_bounded(smem_u32(&sh.full[stage]), phase, abort_flag, XWAIT_NS)) {
          x_fail(sh, p.status);
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t sa = ring + stage * XSTAGE;
        const uint32_t sb = sa + XA_BYTES;
        const uint32_t sf = sfring + stage * XSF_BYTES;
        // this stage's scale slot is free: its previous MMAs completed
        // before the producer could refill the stage
        const uint32_t tsf = tmem + XSF_COL + stage * 8;
        tmem_cp_atom(tsf, sf);
        tmem_cp_atom(tsf + 4, sf + kMxAtom);
#pragma unroll
        for (int kk = 0; kk < XBK / XUK; ++kk) {
          const uint64_t ad = umma_desc_sw128(sa + kk * XUK, 16, 1024);
          const uint64_t bd = umma_desc_sw128(sb + kk * XUK, 16, 1024);
          umma_mx(d_tmem, ad, bd, umma_idesc_sfid(idesc0, (uint32_t)kk), tsf, tsf + 4,
                  (kb | kk) != 0 ? 1u : 0u);
        }
        umma_commit(smem_u32(&sh.empty[stage]));
        if (++stage == XSTAGES) { stage = 0; phase ^= 1u; }
      }
      if (!ok) break;
      umma_commit(smem_u32(&sh.tfull[acc]));
    }
    // all issued MMAs complete before TMEM can be released
    umma_commit(smem_u32(&sh.drain));
    int dummy = 0;
    mbar_wait_bounded(smem_u32(&sh.drain), 0, &dummy, XDRAIN_NS);
  } else if (warp >= XEPI0) {
    // ---------------- epilogue: TMEM lanes 32*(warp%4) .. +31, column half
    const int q = warp & 3;
    const int half = (warp - XEPI0) >> 2;
    int it = 0;
    for (int idx = blockIdx.x; idx < ntiles; idx += gridDim.x, ++it) {
      const XTile t = x_tile<KIND>(p, sh, idx);
      const int acc = it & 1;
      const uint32_t acc_phase = (it >> 1) & 1;
      if (!mbar_wait_bounded(smem_u32(&sh.tfull[acc]), acc_phase, abort_flag, XWAIT_NS)) {
        if (lane == 0) x_fail(sh, p.status);
        break;
      }
      tc_fence_after();
      const uint32_t tacc = tmem + ((uint32_t)(q * 32) << 16) + acc * XBN;
      const int row = t.m0 + q * 32 + lane;
      uint32_t r0[32], r1[32];
      if (KIND == MXK_GATE_UP) {
        // 32 hidden units per half: gate columns half*32.., up columns 64 + half*32..
        tmem_ld32(tacc + half * 32, r0);
        tmem_ld32(tacc + XBN / 2 + half * 32, r1);
        tmem_ld_wait();
        tc_fence_before();
        mbar_arrive(smem_u32(&sh.tempty[acc]));    // accumulator free once in registers
        float h[32];
#pragma unroll
        for (int i = 0; i < 32; ++i)
          h[i] = x_silu(__uint_as_float(r0[i])) * __uint_as_float(r1[i]);
        uint32_t cq[8];
        const uint32_t sbyte = mx_quant32(h, cq);
        const int col = t.n0 + half * 32;
        uint8_t* o = p.hq + (size_t)row * p.H + col;
        st_v4(o, make_uint4(cq[0], cq[1], cq[2], cq[3]));
        st_v4(o + 16, make_uint4(cq[4], cq[5], cq[6], cq[7]));
        p.hs[((size_t)(row >> 7) * (p.H / 128) + (col >> 7)) * kMxAtom +
             mx_sf_byte(row & 127, (col >> 5) & 3)] = (uint8_t)sbyte;
      } else {
        // 64 model columns per half, fp32
        tmem_ld32(tacc + half * 64, r0);
        tmem_ld32(tacc + half * 64 + 32, r1);
        tmem_ld_wait();
        tc_fence_before();
        mbar_arrive(smem_u32(&sh.tempty[acc]));
        float* o = p.out + (size_t)row * p.d + t.n0 + half * 64;
#pragma unroll
        for (int i = 0; i < 8; ++i)
          st_v4(o + 4 * i, make_uint4(r0[4 * i], r0[4 * i + 1], r0[4 * i + 2], r0[4 * i + 3]));
#pragma unroll
        for (int i = 0; i < 8; ++i)
          st_v4(o + 32 + 4 * i,
                make_uint4(r1[4 * i], r1[4 * i + 1], r1[4 * i + 2], r1[4 * i + 3]));
      }
    }
  }
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (warp == 2) {
    tc_fence_after();
    tmem_dealloc(tmem, XTMEM_COLS);
  }
}

// ------------------------------------------------------------------ weights
// One thread per block of 32 along K of one weight row: codes stay in the
// row's place ([rows][K]); the scale byte goes to the atom of the row's tile
// row.  Gate/up (W_gu [E][2H][d]): tile block jb = n / 64 of the hidden units
// holds gate rows 64 jb.. at tile rows 0-63 and the matching up rows at
// 64-127.  Down (W_down [E][d][H]): tile block jb = n / 128, tile row n % 128.
__global__ void __launch_bounds__(256)
mx_quant_weights_kernel(const bf16* __restrict__ W, uint8_t* __restrict__ Wq,
                        uint8_t* __restrict__ Ws, long long rows, int K, int rows_per_e,
                        int gate_up, int H) {
  const int nb = K / 32, kg = K / 128;
  const long long total = rows * nb;
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < total;
       i += (long long)gridDim.x * blockDim.x) {
    const long long row = i / nb;
    const int b = (int)(i - row * nb);
    const bf16* src = W + row * K + b * 32;
    float v[32];
#pragma unroll
    for (int u = 0; u < 4; ++u) unpack8(ld_nc_v4(src + u * 8), v + 8 * u);
    uint32_t cq[8];
    const uint32_t sbyte = mx_quant32(v, cq);
    uint8_t* o = Wq + row * K + b * 32;
    st_v4(o, make_uint4(cq[0], cq[1], cq[2], cq[3]));
    st_v4(o + 16, make_uint4(cq[4], cq[5], cq[6], cq[7]));
    const int e = (int)(row / rows_per_e);
    const int n = (int)(row - (long long)e * rows_per_e);
    int jb, v_row, nbt;
    if (gate_up) {
      const bool up = n >= H;
      const int nn = up ? n - H : n;
      jb = nn / 64;
      v_row = nn % 64 + (up ? 64 : 0);
      nbt = H / 64;
    } else {
      jb = n / 128;
      v_row = n % 128;
      nbt = rows_per_e / 128;
    }
    Ws[(((size_t)e * nbt + jb) * kg + (b >> 2)) * kMxAtom + mx_sf_byte(v_row, b & 3)] =
        (uint8_t)sbyte;
  }
}


// ------------------------------------------------------------------ host side
typedef CUresult (*XEncodeFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                              const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                              const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                              CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

XEncodeFn x_encode_fn() {
  static XEncodeFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                         cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<XEncodeFn>(ptr);
  });
  return fn;
}

// Byte tensor map (e4m3 codes), 128-byte swizzle, zero fill out of bounds.
// dims innermost first; strides in bytes for dims 1..rank-1.
bool x_make_map(CUtensorMap* m, const void* ptr, int rank, const uint64_t* dims,
                const uint64_t* strides, const uint32_t* box) {
  XEncodeFn fn = x_encode_fn();
  if (!fn) return false;
  cuuint64_t gd[5], gs[4];
  cuuint32_t bx[5], es[5];
  for (int i = 0; i < rank; ++i) { gd[i] = dims[i]; bx[i] = box[i]; es[i] = 1; }
  for (int i = 0; i < rank - 1; ++i) gs[i] = strides[i];
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, (cuuint32_t)rank, const_cast<void*>(ptr), gd, gs,
            bx, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int KIND>
cudaError_t x_launch(const CUtensorMap& a, const CUtensorMap& b, const XParams& p, int sms,
                     cudaStream_t s) {
  static std::once_flag once;
  static cudaError_t err = cudaSuccess;
  std::call_once(once, [] {
    err = cudaFuncSetAttribute(mx_gemm_kernel<KIND>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               (int)XSMEM);
  });
  if (err != cudaSuccess) return err;
  mx_gemm_kernel<KIND><<<sms, XTHREADS, XSMEM, s>>>(a, b, p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_mx_gemm(const MxGemmCall& g, cudaStream_t s) {
  DeviceInfo di;
  if (device_info(&di) != MOE_OK) return cudaErrorUnknown;
  XParams p{};
  p.row_offsets = g.row_offsets;
  p.E = g.E;
  p.H = g.H;
  p.d = g.d;
  p.sfa = g.sfa;
  p.sfb = g.sfb;
  p.hq = g.hq;
  p.hs = g.hs;
  p.out = g.out;
  p.status = g.status;
  CUtensorMap ta, tb;
  const uint64_t rows = (uint64_t)g.rows;
  bool ok;
  if (g.gate_up) {
    // A: x codes [rows][d]; B: W_gu codes [E][2][H][d] -> dims {d, H, 2, E}
    p.K = g.d;
    p.n_tiles = g.H / (XBN / 2);
    p.nbt = g.H / (XBN / 2);
    uint64_t da[2] = {(uint64_t)g.d, rows}, sa[1] = {(uint64_t)g.d};
    uint32_t ba[2] = {XBK, XBM};
    uint64_t db[4] = {(uint64_t)g.d, (uint64_t)g.H, 2, (uint64_t)g.E};
    uint64_t sb[3] = {(uint64_t)g.d, (uint64_t)g.H * g.d, (uint64_t)2 * g.H * g.d};
    uint32_t bb[4] = {XBK, XBN / 2, 1, 1};
    ok = x_make_map(&ta, g.A, 2, da, sa, ba) && x_make_map(&tb, g.B, 4, db, sb, bb);
  } else {
    // A: h codes [rows][H]; B: W_down codes [E][d][H] -> dims {H, d, E}
    p.K = g.H;
    p.n_tiles = g.d / XBN;
    p.nbt = g.d / XBN;
    uint64_t da[2] = {(uint64_t)g.H, rows}, sa[1] = {(uint64_t)g.H};
    uint32_t ba[2] = {XBK, XBM};
    uint64_t db[3] = {(uint64_t)g.H, (uint64_t)g.d, (uint64_t)g.E};
    uint64_t sb[2] = {(uint64_t)g.H, (uint64_t)g.d * g.H};
    uint32_t bb[3] = {XBK, XBN, 1};
    ok = x_make_map(&ta, g.A, 2, da, sa, ba) && x_make_map(&tb, g.B, 3, db, sb, bb);
  }
  if (!ok) return cudaErrorInvalidValue;
  p.kg = p.K / XBK;
  return g.gate_up ? x_launch<MXK_GATE_UP>(ta, tb, p, di.num_sms, s)
                   : x_launch<MXK_DOWN>(ta, tb, p, di.num_sms, s);
}

cudaError_t launch_mx_quant_weights(const moe_config& c, const void* W_gu, const void* W_down,
                                    uint8_t* W_gu_q, uint8_t* W_gu_s, uint8_t* W_down_q,
                                    uint8_t* W_down_s, cudaStream_t s) {
  DeviceInfo di;
  if (device_info(&di) != MOE_OK) return cudaErrorUnknown;
  const int grid = di.num_sms * 8;
  mx_quant_weights_kernel<<<grid, 256, 0, s>>>(static_cast<const bf16*>(W_gu), W_gu_q, W_gu_s,
                                               (long long)c.E * 2 * c.H, c.d, 2 * c.H, 1, c.H);
  mx_quant_weights_kernel<<<grid, 256, 0, s>>>(static_cast<const bf16*>(W_down), W_down_q,
                                               W_down_s, (long long)c.E * c.d, c.H, c.d, 0, c.H);
  return cudaGetLastError();
}

}  // namespace moe
