// MXFP8 experts on the 5th-generation tensor cores (sm_103a).
//
// "KohakUwULLM" README, Key features and Selected measurements: MXFP8 (e4m3
// values, UE8M0 scales per 32 values) on the feed-forward pair and the routed
// experts, with fully fused expert kernels that never materialise the
// (tokens * top_k, hidden) intermediates in 16-bit form.
//
// Here that is:
//   * a row quantiser (bf16 weights, or x in token order for the shared
//     expert -> e4m3 codes + scale atoms);
//   * the quantising permute (moe_dispatch.cu, perm_scatter_kernel<true>);
//   * a persistent grouped GEMM on CTA pairs with tcgen05.mma.cta_group::2
//     .kind::mxf8f6f4 and block scales.  A pair computes a 256 x 256 tile:
//     each CTA loads (TMA, 128-byte swizzle) its 128 rows of A and half of
//     the 256 B rows, plus three 512-byte scale atoms -- its own rows' A
//     scales and the scales of all 256 B rows, which both CTAs need -- all
//     completing on the even CTA's barrier.  The even CTA's MMA thread moves
//     both CTAs' atoms into their TMEM with tcgen05.cp.cta_group::2 and issues
//     four K = 32 MMAs per stage, each picking its K-block's scale byte by the
//     scale-factor id;
//   * epilogues: gate/up -> h = silu(a) * b quantised straight to MXFP8 (codes
//     and scale atoms of h, no bf16 h); down -> out_perm (routed) or s_out
//     (the shared expert, the same kernel over dense token rows), fp32, for
//     the combine.
// Per CTA: one 256-column accumulator (the scale slots of the six 34 KB
// stages take TMEM columns 256-351, so a second accumulator does not fit);
// the epilogue warps pull the accumulator into registers and release it
// before their arithmetic, so the MMAs of the next tile wait only for that
// drain.  The tile shape is set by load traffic: at fp8 rates the L2 -> SM
// bytes per flop decide the pace (256 x 128 pair tiles were bound by about
// 13 TB/s of loads), and 256 x 256 pair tiles halve them.
#include <algorithm>
#include <cstring>
#include <mutex>

#include <cuda_fp16.h>

#include "moe_common.cuh"
#include "moe_internal.h"
#include "moe_mx.cuh"

namespace moe {

namespace {

constexpr int XBM = 128;                    // tile rows per CTA (256 per pair)
constexpr int XBN = 256;                    // tile columns (UMMA N of the pair)
constexpr int XBK = 128;                    // K per stage: one 128-byte row of e4m3
constexpr int XUK = 32;                     // K per MMA (= one scale block)
constexpr int XA_BYTES = XBM * XBK;         // 16 KB: this CTA's A rows
constexpr int XB_BYTES = (XBN / 2) * XBK;   // 16 KB: this CTA's half of the B rows
constexpr int XSF_OFF = XA_BYTES + XB_BYTES;
constexpr int XLOAD = XSF_OFF + 3 * kMxAtom;    // + A atom, two B atoms: bytes per CTA and stage
constexpr int XSTAGE = 34 * 1024;               // stage stride (1024-byte aligned)
constexpr int XSTAGES = 6;
constexpr int XTHREADS = 384;               // warp 0 TMA, 1 MMA, 2 TMEM, 3 scan, 4-11 epilogue
constexpr int XEPI0 = 4;
constexpr int XEPI_WARPS = 8;
constexpr int XTMEM_COLS = 512;
constexpr int XSF_COL = XBN;                // stage s scales: columns 256 + 16 s (A), + 4, + 8 (B)
constexpr int XSF_SLOT = 16;
constexpr uint64_t XWAIT_NS = 2000000000ull;  // bounded waits give up after 2 s
constexpr uint64_t XDRAIN_NS = 200000000ull;
constexpr size_t XRESERVE = 3072;           // struct XShared
// dH epilogue: each thread's two prefetch slots for its row's a | b chunks
// (64 + 64 bytes, padded to 144 so that the rows of a warp fall on distinct
// banks for 16-byte accesses)
constexpr int XPRE_ROW = 144;

// MXK_GATE_UP_SAVE: gate/up that also stores h in bf16 and a | b in fp16
// (training)
enum MxKind { MXK_GATE_UP = 0, MXK_DOWN = 1, MXK_DH = 2, MXK_GATE_UP_SAVE = 3 };
template <int KIND>
struct XIsGateUp {
  static constexpr bool value = KIND == MXK_GATE_UP || KIND == MXK_GATE_UP_SAVE;
};
// Pipeline depth and shared memory by kind: the dH kernel gives two stages
// to the epilogue's a | b prefetch slots.
template <int KIND>
struct XCfg {
  static constexpr int stages = KIND == MXK_DH ? 4 : XSTAGES;
  static constexpr size_t pre = KIND == MXK_DH ? (size_t)XEPI_WARPS * 2 * 32 * XPRE_ROW : 0;
  static constexpr size_t smem = XRESERVE + 1024 + (size_t)stages * XSTAGE + pre;
  static_assert(smem <= 232448, "exceeds the 227 KB opt-in shared memory of a block");
};
static_assert(XSTAGE % 1024 == 0 && XLOAD <= XSTAGE, "stage layout");
static_assert(XSF_COL + XSF_SLOT * XSTAGES <= XTMEM_COLS, "scale slots exceed TMEM");

struct XParams {
  const int32_t* row_offsets;  // [E+1] padded segment offsets (multiples of 128), or NULL:
                               // dense rows (one group of dense_rows rows, E = 1)
  int dense_rows;
  int row_limit;               // rows at or past it are not stored
  int E;
  int H;                       // hidden size (gate/up: output units; down: K)
  int d;                       // model dim
  int n_tiles;                 // column tiles per pair of 128-row blocks
  int kg;                      // K / 128: scale atoms per row block
  int nbt;                     // weight scale blocks (128 rows) per expert
  uint8_t* hq;                 // gate/up: h codes [R][H]
  uint8_t* hs;                 // gate/up: h scale atoms [R/128][H/128][512]
  bf16* hb;                    // gate/up, training: h [R][H] bf16, or NULL
  __half* abo;                 // gate/up, training: a | b [R][2H] fp16, or NULL
  void* out;                   // down: [rows][d], fp32 or (out_bf16) bf16
  int out_bf16;
  const __half* abi;           // dH: the saved a | b [R][2H] fp16
  bf16* dgu;                   // dH: d_gu = da | db [R][2H] bf16
  uint8_t* dgq;                // dH: codes of d_gu [R][2H]
  uint8_t* dgs;                // dH: scale atoms of d_gu [R/128][2H/128][512]
  int* status;
};

struct XShared {
  uint64_t full[XSTAGES];
  uint64_t empty[XSTAGES];
  uint64_t tfull;
  uint64_t tempty;
  uint64_t drain;
  uint32_t tmem_base;
  int abort_flag;
  int roff[257];               // padded segment offsets
  int ppre[257];               // 256-row pair tiles before expert e
  int roff_bad;                // debug builds: the segment table failed its check
};
static_assert(sizeof(XShared) <= XRESERVE, "bookkeeping too large");

struct XTile {
  int e, m0, n0, row_end;      // m0: the pair's first row
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

// Tile idx: pair unit idx / n_tiles (two 128-row blocks of one expert's
// padded segment; an odd last block is paired with the block after the
// segment, computed and not stored), column tile idx % n_tiles (128 hidden
// units = 128 gate + 128 up weight rows for gate/up, 256 model columns for
// down).
template <int KIND>
__device__ __forceinline__ XTile x_tile(const XParams& p, const XShared& sh, int idx) {
  XTile t;
  const int mu = idx / p.n_tiles;
  t.n0 = (idx - mu * p.n_tiles) * (XIsGateUp<KIND>::value ? XBN / 2 : XBN);
  t.e = x_last_le(sh.ppre, p.E, mu);
  t.m0 = sh.roff[t.e] + (mu - sh.ppre[t.e]) * 2 * XBM;
  t.row_end = sh.roff[t.e + 1];
  return t;
}

__device__ __forceinline__ void x_fail(XShared& sh, int* status) {
  set_status(status, MOE_ERR_TIMEOUT);
  *(volatile int*)&sh.abort_flag = 1;
}

// The logistic function with CUDA's fast exponential and approximate
// division; the result is quantised to e4m3 (3 mantissa bits) right after.
__device__ __forceinline__ float x_silu(float a) { return __fdividef(a, 1.f + __expf(-a)); }
__device__ __forceinline__ float x_sigmoid(float a) { return __fdividef(1.f, 1.f + __expf(-a)); }

// 32 consecutive bf16 values: four 16-byte stores.
__device__ __forceinline__ void x_st32(bf16* p, const float* v) {
#pragma unroll
  for (int u = 0; u < 4; ++u) st_v4(p + 8 * u, pack8(v + 8 * u));
}
// Two fp32 values as an fp16 pair (round to nearest even), magnitudes past
// the largest finite fp16 (65504) clamped to it; NaN stays NaN.
__device__ __forceinline__ uint32_t x_f16x2(float lo, float hi) {
  lo = fabsf(lo) > 65504.f ? copysignf(65504.f, lo) : lo;
  hi = fabsf(hi) > 65504.f ? copysignf(65504.f, hi) : hi;
  const __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&h);
}
// 32 fp32 values given as their bits, stored as fp16: two 32-byte stores
// (p 32-byte aligned).
__device__ __forceinline__ void x_st32_f16(__half* p, const uint32_t* r) {
  uint32_t w[16];
#pragma unroll
  for (int u = 0; u < 16; ++u) w[u] = x_f16x2(__uint_as_float(r[2 * u]), __uint_as_float(r[2 * u + 1]));
  st_v8(p, w);
  st_v8(p + 16, w + 8);
}
__device__ __forceinline__ float x_f16_at(const uint32_t* w, int i) {
  const __half2 h = *reinterpret_cast<const __half2*>(&w[i >> 1]);
  return (i & 1) ? __high2float(h) : __low2float(h);
}

// The a | b chunk [col, col + 32) of one row (64 + 64 bytes of fp16) into
// this thread's prefetch slot with asynchronous 16-byte copies (registers
// stay free), as one commit group; an empty group when the row has none.
__device__ __forceinline__ void x_prefetch_ab(bool work, const __half* abi, int H, int row,
                                              int col, uint32_t slot) {
  if (work) {
    const __half* a = abi + (size_t)row * 2 * H + col;
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(slot + 16 * u),
                   "l"(a + 8 * u) : "memory");
      asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(slot + 64 + 16 * u),
                   "l"(a + H + 8 * u) : "memory");
    }
  }
  asm volatile("cp.async.commit_group;" ::: "memory");
}
template <int N>
__device__ __forceinline__ void x_prefetch_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}
__device__ __forceinline__ void ld_shared_v4(uint32_t a, uint32_t* v) {
  asm volatile("ld.shared.v4.b32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]) : "r"(a) : "memory");
}
__device__ __forceinline__ void st_shared_v4(uint32_t a, const uint32_t* v) {
  asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};"
               :: "r"(a), "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]) : "memory");
}

// dH -> the SwiGLU chain rule for 32 columns [col, col + 32) of one row:
// da = dH b s(a) (1 + a (1 - s(a))) and db = dH silu(a) from the saved fp16
// a | b, prefetched into this thread's ``slot``.  Each fp32 result is quantised along 2H (blocks of 32, which never
// straddle da and db: H is a multiple of 128) for the dX product, and stored
// in bf16 as d_gu = da | db for the weight-gradient product: one rounding
// each.  da first, then db, so that one 32-value array is live at a time.
__device__ __forceinline__ void x_dh_chunk(const XParams& p, int row, int col,
                                           const uint32_t* acc, uint32_t slot) {
  const size_t rb = (size_t)row * 2 * p.H;
  const size_t atom_row = (size_t)(row >> 7) * (2 * p.H / 128);
  float v[32];
  uint32_t cq[8];
  // eight values at a time from the slot, so that little of a | b is live;
  // silu(a) = a s(a) of those eight goes back into the 32 slot bytes they
  // came from (fp32), so that db needs no second logistic
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    uint32_t ah[4], bh[4], sl[8];
    ld_shared_v4(slot + 16 * u, ah);
    ld_shared_v4(slot + 64 + 16 * u, bh);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const float a = x_f16_at(ah, i), sg = x_sigmoid(a);
      v[8 * u + i] = __uint_as_float(acc[8 * u + i]) * x_f16_at(bh, i) * sg * (1.f + a * (1.f - sg));
      sl[i] = __float_as_uint(a * sg);
    }
    st_shared_v4(slot + 16 * u, sl);
    st_shared_v4(slot + 64 + 16 * u, sl + 4);
  }
  uint32_t sbyte = mx_quant32(v, cq);
  st_v8(p.dgq + rb + col, cq);
  p.dgs[(atom_row + (col >> 7)) * kMxAtom + mx_sf_byte(row & 127, (col >> 5) & 3)] =
      (uint8_t)sbyte;
  x_st32(p.dgu + rb + col, v);
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    uint32_t sl[8];
    ld_shared_v4(slot + 16 * u, sl);
    ld_shared_v4(slot + 64 + 16 * u, sl + 4);
#pragma unroll
    for (int i = 0; i < 8; ++i) v[8 * u + i] = __uint_as_float(acc[8 * u + i]) * __uint_as_float(sl[i]);
  }
  sbyte = mx_quant32(v, cq);
  st_v8(p.dgq + rb + p.H + col, cq);
  p.dgs[(atom_row + ((p.H + col) >> 7)) * kMxAtom +
        mx_sf_byte(row & 127, ((p.H + col) >> 5) & 3)] = (uint8_t)sbyte;
  x_st32(p.dgu + rb + p.H + col, v);
}

// ------------------------------------------------------------------ kernel
// CTAs run in clusters of two.  Both load their shares of each stage
// (completing on the even CTA's full barrier, which that CTA arms for both);
// the even CTA's MMA thread issues the pair MMAs, whose commits arrive on both
// CTAs' empty and accumulator-full barriers; both CTAs' epilogue warps arrive
// on the even CTA's accumulator-empty barrier once the accumulator is in
// their registers.
template <int KIND>
__global__ void __launch_bounds__(XTHREADS, 1)
mx_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
               const __grid_constant__ CUtensorMap tmSA, const __grid_constant__ CUtensorMap tmSB,
               const XParams p) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t ring = (raw + (uint32_t)XRESERVE + 1023u) & ~1023u;
  // both CTAs of a pair see the same layout, so both return here together
  constexpr int kStages = XCfg<KIND>::stages;
  if (ring + (uint32_t)(kStages * XSTAGE + XCfg<KIND>::pre) - raw > (uint32_t)XCfg<KIND>::smem) {
    if (threadIdx.x == 0) set_status(p.status, MOE_ERR_DEVICE);
    return;
  }
  XShared& sh = *reinterpret_cast<XShared*>(smem_raw);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int rank = (int)cluster_ctarank();
  const int unit = (int)(blockIdx.x >> 1);
  const int nunits = (int)(gridDim.x >> 1);

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(smem_u32(&sh.full[s]), 1);
      mbar_init(smem_u32(&sh.empty[s]), 1);
    }
    mbar_init(smem_u32(&sh.tfull), 1);
    mbar_init(smem_u32(&sh.tempty), 2 * XEPI_WARPS);
    mbar_init(smem_u32(&sh.drain), 1);
    sh.abort_flag = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
    tma_prefetch_desc(&tmSA);
    tma_prefetch_desc(&tmSB);
  }
  if (p.row_offsets) {
    for (int e = threadIdx.x; e <= p.E; e += blockDim.x) sh.roff[e] = p.row_offsets[e];
  } else if (threadIdx.x == 0) {
    sh.roff[0] = 0;
    sh.roff[1] = (p.dense_rows + XBM - 1) / XBM * XBM;
  }
  if (warp == 2) {
    tmem_alloc_pair(smem_u32(&sh.tmem_base), XTMEM_COLS);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  __syncthreads();
  if (kDebugBounds && p.row_offsets && threadIdx.x == 0) {
    sh.roff_bad = dbg_roff_ok(sh.roff, p.E, p.row_limit) ? 0 : 1;
    if (sh.roff_bad) set_status(p.status, MOE_ERR_BOUNDS);
  }
  if (warp == 3) {
    // 256-row pair tiles per expert, prefix over experts
    int carry = 0;
    for (int e0 = 0; e0 < p.E; e0 += 32) {
      const int e = e0 + lane;
      int v = e < p.E ? ((sh.roff[e + 1] - sh.roff[e]) / XBM + 1) / 2 : 0;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += y;
      }
      if (e < p.E) sh.ppre[e + 1] = carry + v;
      carry += __shfl_sync(0xffffffffu, v, 31);
    }
    if (lane == 0) sh.ppre[0] = 0;
  }
  // barriers of both CTAs initialised and ppre visible before any signal
  cluster_sync();
  tc_fence_after();
  const uint32_t tmem = sh.tmem_base;
  volatile int* abort_flag = &sh.abort_flag;
  const int ntiles = (kDebugBounds && p.row_offsets && sh.roff_bad) ? 0 : sh.ppre[p.E] * p.n_tiles;

  if (warp == 0 && lane == 0) {
    // ---------------- producer (both CTAs)
    int stage = 0;
    uint32_t phase = 0;
    bool ok = true;
    for (int idx = unit; idx < ntiles && ok; idx += nunits) {
      const XTile t = x_tile<KIND>(p, sh, idx);
      const int rowA = t.m0 + XBM * rank;
      // the tile's two 128-row weight blocks: gate and up rows of the same
      // hidden units (gate/up), or two consecutive blocks of model columns
      const int jb0 = t.n0 / 128;
      const int jb1 = XIsGateUp<KIND>::value ? (p.H + t.n0) / 128 : t.n0 / 128 + 1;
      const int atom_a = (rowA / XBM) * p.kg;                 // this CTA's rows' scales
      const int atom_b0 = (t.e * p.nbt + jb0) * p.kg;
      const int atom_b1 = (t.e * p.nbt + jb1) * p.kg;
      for (int kb = 0; kb < p.kg; ++kb) {
        if (!mbar_wait_bounded(smem_u32(&sh.empty[stage]), phase ^ 1u, abort_flag, XWAIT_NS)) {
          x_fail(sh, p.status);
          ok = false;
          break;
        }
        const uint32_t fb_local = smem_u32(&sh.full[stage]);
        const uint32_t fb = mapa_shared(fb_local, 0);
        if (rank == 0) mbar_arrive_expect_tx(fb_local, 2 * XLOAD);
        const uint32_t sa = ring + stage * XSTAGE;
        const uint32_t sb = sa + XA_BYTES;
        const uint32_t sf = sa + XSF_OFF;
        tma_load_2d_pair(sa, &tmA, fb, kb * XBK, rowA);
        if (XIsGateUp<KIND>::value)   // rank 0: the 128 gate rows, rank 1: the 128 up rows
          tma_load_4d_pair(sb, &tmB, fb, kb * XBK, t.n0, rank, t.e);
        else
          tma_load_3d_pair(sb, &tmB, fb, kb * XBK, t.n0 + (XBN / 2) * rank, t.e);
        tma_load_2d_pair(sf, &tmSA, fb, 0, (atom_a + kb) * 4);
        tma_load_2d_pair(sf + kMxAtom, &tmSB, fb, 0, (atom_b0 + kb) * 4);
        tma_load_2d_pair(sf + 2 * kMxAtom, &tmSB, fb, 0, (atom_b1 + kb) * 4);
        if (++stage == kStages) { stage = 0; phase ^= 1u; }
      }
    }
    if (!ok) {
      // this CTA's copies complete on the even CTA's barriers: give the ones
      // in flight a bounded time to land before shared memory is released
      const uint64_t t0 = global_ns();
      while (global_ns() - t0 < XDRAIN_NS) {
      }
    }
  } else if (warp == 1 && lane == 0 && rank == 0) {
    // ---------------- MMA issuer (even CTA)
    constexpr uint32_t idesc0 = umma_idesc_mx(2 * XBM, XBN);
    int stage = 0;
    uint32_t phase = 0;
    int it = 0;
    bool ok = true;
    for (int idx = unit; idx < ntiles && ok; idx += nunits, ++it) {
      if (!mbar_wait_bounded_cluster(smem_u32(&sh.tempty), (it & 1) ^ 1u, abort_flag,
                                     XWAIT_NS)) {
        x_fail(sh, p.status);
        break;
      }
      tc_fence_after();
      for (int kb = 0; kb < p.kg; ++kb) {
        if (!mbar_wait_bounded(smem_u32(&sh.full[stage]), phase, abort_flag, XWAIT_NS)) {
          x_fail(sh, p.status);
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t sa = ring + stage * XSTAGE;
        const uint32_t sb = sa + XA_BYTES;
        const uint32_t sf = sa + XSF_OFF;
        // this stage's scale slot is free in both CTAs: its previous MMAs
        // completed before either producer could refill the stage
        const uint32_t tsf = tmem + XSF_COL + stage * XSF_SLOT;
        tmem_cp_atom_pair(tsf, sf);
        tmem_cp_atom_pair(tsf + 4, sf + kMxAtom);
        tmem_cp_atom_pair(tsf + 8, sf + 2 * kMxAtom);
#pragma unroll
        for (int kk = 0; kk < XBK / XUK; ++kk) {
          const uint64_t ad = umma_desc_sw128(sa + kk * XUK, 16, 1024);
          const uint64_t bd = umma_desc_sw128(sb + kk * XUK, 16, 1024);
          umma_mx_pair(tmem, ad, bd, umma_idesc_sfid(idesc0, (uint32_t)kk), tsf, tsf + 4,
                       (kb | kk) != 0 ? 1u : 0u);
        }
        umma_commit_pair(smem_u32(&sh.empty[stage]), 3);
        if (++stage == kStages) { stage = 0; phase ^= 1u; }
      }
      if (!ok) break;
      umma_commit_pair(smem_u32(&sh.tfull), 3);
    }
    // all issued MMAs complete before TMEM can be released
    umma_commit_pair(smem_u32(&sh.drain), 1);
    int dummy = 0;
    mbar_wait_bounded(smem_u32(&sh.drain), 0, &dummy, XDRAIN_NS);
  } else if (warp >= XEPI0) {
    // ---------------- epilogue (both CTAs): TMEM lanes 32*(warp%4) .. +31
    const int q = warp & 3;
    const int half = (warp - XEPI0) >> 2;
    const uint32_t tempty_leader = mapa_shared(smem_u32(&sh.tempty), 0);
    // dH: this thread's two a | b prefetch slots
    const uint32_t pre = ring + (uint32_t)(kStages * XSTAGE) +
                         (uint32_t)(((warp - XEPI0) * 2 * 32 + lane) * XPRE_ROW);
    int it = 0;
    for (int idx = unit; idx < ntiles; idx += nunits, ++it) {
      const XTile t = x_tile<KIND>(p, sh, idx);
      const int blk = t.m0 + XBM * rank;            // this CTA's 128 rows
      const bool store = blk < t.row_end;           // else the pair's padding half
      const int row = blk + q * 32 + lane;
      const bool row_ok = row < p.row_limit;
      const int col0 = t.n0 + half * 128;           // dH: this warp's first column
      const bool work = KIND == MXK_DH && store && row_ok && col0 < p.H;
      if (KIND == MXK_DH) {
        // the first two chunks' a | b, fetched while the MMAs run
        x_prefetch_ab(work, p.abi, p.H, row, col0, pre);
        x_prefetch_ab(work, p.abi, p.H, row, col0 + 32, pre + 32 * XPRE_ROW);
      }
      if (!mbar_wait_bounded(smem_u32(&sh.tfull), it & 1, abort_flag, XWAIT_NS)) {
        if (lane == 0) x_fail(sh, p.status);
        if (KIND == MXK_DH) x_prefetch_wait<0>();
        break;
      }
      tc_fence_after();
      const uint32_t tacc = tmem + ((uint32_t)(q * 32) << 16);
      // this warp's 128 accumulator columns into registers; gate/up: gate
      // columns half*64 .. +63 and the matching up columns 128 + half*64 ..
      uint32_t r[4][32];
      if (XIsGateUp<KIND>::value) {
        tmem_ld64(tacc + half * 64, &r[0][0]);
        tmem_ld64(tacc + XBN / 2 + half * 64, &r[2][0]);
      } else if (KIND == MXK_DH) {
        tmem_ld32(tacc + half * 128, &r[0][0]);     // the first 32 of the 128 columns
      } else {
        tmem_ld128(tacc + half * 128, &r[0][0]);
      }
      tmem_ld_wait();
      if (KIND == MXK_DH) {
        // 64 columns at a time, which keeps the chain rule in registers; the
        // accumulator is released once the second 64 are read, about half
        // way through this (memory-bound) epilogue, well before the next
        // tile's MMAs could finish.  Each chunk's a | b waits in a prefetch
        // slot, refilled with the chunk two ahead as soon as it is read.
        // Column halves past H are the last tile's padding.
        const uint32_t pre1 = pre + 32 * XPRE_ROW;
        x_prefetch_wait<1>();
        if (work) x_dh_chunk(p, row, col0, r[0], pre);
        x_prefetch_ab(work, p.abi, p.H, row, col0 + 64, pre);
        __syncwarp();
        tmem_ld32(tacc + half * 128 + 32, &r[0][0]);
        tmem_ld_wait();
        x_prefetch_wait<1>();
        if (work) x_dh_chunk(p, row, col0 + 32, r[0], pre1);
        x_prefetch_ab(work, p.abi, p.H, row, col0 + 96, pre1);
        __syncwarp();
        tmem_ld64(tacc + half * 128 + 64, &r[0][0]);
        tmem_ld_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_cluster(tempty_leader);
        x_prefetch_wait<1>();
        if (work) x_dh_chunk(p, row, col0 + 64, r[0], pre);
        x_prefetch_wait<0>();
        if (work) x_dh_chunk(p, row, col0 + 96, r[1], pre1);
        continue;
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(tempty_leader);   // accumulator free
      if (!store) continue;
      if (XIsGateUp<KIND>::value) {
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          const int col = t.n0 + half * 64 + c * 32;
          if (KIND == MXK_GATE_UP_SAVE && row_ok) {
            // training: the pre-activations a | b in fp16 for the chain
            // rule, whose results feed an e4m3 quantiser: 11 significant
            // bits keep the codes it moves rare, where bf16's 8 would move
            // about 2% of them by a whole step
            x_st32_f16(p.abo + (size_t)row * 2 * p.H + col, r[c]);
            x_st32_f16(p.abo + (size_t)row * 2 * p.H + p.H + col, r[2 + c]);
          }
          float h[32];
#pragma unroll
          for (int i = 0; i < 32; ++i)
            h[i] = x_silu(__uint_as_float(r[c][i])) * __uint_as_float(r[2 + c][i]);
          uint32_t cq[8];
          const uint32_t sbyte = mx_quant32(h, cq);
          if (row_ok) {
            st_v8(p.hq + (size_t)row * p.H + col, cq);
            p.hs[((size_t)(row >> 7) * (p.H / 128) + (col >> 7)) * kMxAtom +
                 mx_sf_byte(row & 127, (col >> 5) & 3)] = (uint8_t)sbyte;
            // training: h in bf16 as well (the weight-gradient product's)
            if (KIND == MXK_GATE_UP_SAVE) x_st32(p.hb + (size_t)row * p.H + col, h);
          }
        }
      } else {
        const size_t o0 = (size_t)row * p.d + t.n0 + half * 128;
        if (row_ok && p.out_bf16) {
          // the per-slot rows (out_perm, dx_perm) in bf16: 64 bytes per chunk
          bf16* o = static_cast<bf16*>(p.out) + o0;
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            uint32_t w[16];
#pragma unroll
            for (int u = 0; u < 16; ++u)
              w[u] = pack_bf16(__uint_as_float(r[c][2 * u]), __uint_as_float(r[c][2 * u + 1]));
            st_v8(o + 32 * c, w);
            st_v8(o + 32 * c + 16, w + 8);
          }
        } else if (row_ok) {
          float* o = static_cast<float*>(p.out) + o0;
#pragma unroll
          for (int c = 0; c < 4; ++c)
#pragma unroll
            for (int i = 0; i < 4; ++i) st_v8(o + 32 * c + 8 * i, &r[c][8 * i]);
        }
      }
    }
  }
  __syncwarp();
  tc_fence_before();
  // no CTA of a pair leaves (or frees TMEM) while its peer may still signal
  // its barriers or the pair's MMAs may still write its TMEM
  cluster_sync();
  if (warp == 2) {
    tc_fence_after();
    tmem_dealloc_pair(tmem, XTMEM_COLS);
  }
}

// ------------------------------------------------------------------ rows
// One thread per block of 32 along K of one row of a [rows][K] bf16 matrix:
// codes stay in the row's place; the scale byte goes to the atom of the row's
// 128-row block of its group (rows_per_group rows each: an expert's W_gu or
// W_down, or all of x).  Rows at or past rows_real, and rows with valid == 0,
// quantise as zeros (x's padding to 128 rows and its PAD tokens).
__global__ void __launch_bounds__(256)
mx_quant_rows_kernel(const bf16* __restrict__ W, uint8_t* __restrict__ Wq,
                     uint8_t* __restrict__ Ws, long long rows, long long rows_real, int K,
                     int rows_per_group, const uint8_t* __restrict__ valid) {
  const int nb = K / 32, kg = K / 128, nbt = rows_per_group / 128;
  const long long total = rows * nb;
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < total;
       i += (long long)gridDim.x * blockDim.x) {
    const long long row = i / nb;
    const int b = (int)(i - row * nb);
    float v[32];
    if (row < rows_real && !(valid && valid[row] == 0)) {
      const bf16* src = W + row * K + b * 32;
#pragma unroll
      for (int u = 0; u < 4; ++u) unpack8(ld_nc_v4(src + u * 8), v + 8 * u);
    } else {
#pragma unroll
      for (int u = 0; u < 32; ++u) v[u] = 0.f;
    }
    uint32_t cq[8];
    const uint32_t sbyte = mx_quant32(v, cq);
    st_v8(Wq + row * K + b * 32, cq);
    const int e = (int)(row / rows_per_group);
    const int n = (int)(row - (long long)e * rows_per_group);
    Ws[(((size_t)e * nbt + n / 128) * kg + (b >> 2)) * kMxAtom + mx_sf_byte(n % 128, b & 3)] =
        (uint8_t)sbyte;
  }
}

// ------------------------------------------------------------------ columns
// One thread per (group g, column c, block rb of 32 rows) of W [G][R][C]
// bf16: the block W[g][32 rb .. 32 rb + 31][c] (consecutive threads read
// consecutive columns, so each row's loads are coalesced) becomes 32 codes
// of row c of the transpose, Wq[g][c][32 rb ..], and one scale byte in the
// atom of (row block c / 128, K group rb / 4) of group g.
__global__ void __launch_bounds__(256)
mx_quant_cols_kernel(const bf16* __restrict__ W, uint8_t* __restrict__ Wq,
                     uint8_t* __restrict__ Ws, int G, int R, int C) {
  const int nrb = R / 32, kg = R / 128, nbt = C / 128;
  const long long total = (long long)G * nrb * C;
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < total;
       i += (long long)gridDim.x * blockDim.x) {
    const int c = (int)(i % C);
    const long long gr = i / C;
    const int rb = (int)(gr % nrb);
    const int g = (int)(gr / nrb);
    const bf16* src = W + ((size_t)g * R + (size_t)rb * 32) * C + c;
    float v[32];
#pragma unroll
    for (int u = 0; u < 32; ++u) v[u] = __bfloat162float(src[(size_t)u * C]);
    uint32_t cq[8];
    const uint32_t sbyte = mx_quant32(v, cq);
    st_v8(Wq + ((size_t)g * C + c) * R + (size_t)rb * 32, cq);
    Ws[(((size_t)g * nbt + c / 128) * kg + (rb >> 2)) * kMxAtom + mx_sf_byte(c % 128, rb & 3)] =
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

// Byte tensor map, zero fill out of bounds; dims innermost first, strides in
// bytes for dims 1..rank-1.  Codes use the 128-byte swizzle; scale atoms are
// copied as plain 4 x 128-byte boxes.
bool x_make_map(CUtensorMap* m, const void* ptr, int rank, const uint64_t* dims,
                const uint64_t* strides, const uint32_t* box, bool swizzle) {
  XEncodeFn fn = x_encode_fn();
  if (!fn) return false;
  cuuint64_t gd[5], gs[4];
  cuuint32_t bx[5], es[5];
  for (int i = 0; i < rank; ++i) { gd[i] = dims[i]; bx[i] = box[i]; es[i] = 1; }
  for (int i = 0; i < rank - 1; ++i) gs[i] = strides[i];
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, (cuuint32_t)rank, const_cast<void*>(ptr), gd, gs,
            bx, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
            swizzle ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Scale atoms [n_atoms][512] as a [4 n_atoms][128] byte matrix, one atom per box.
bool x_atom_map(CUtensorMap* m, const void* ptr, size_t n_atoms) {
  uint64_t dims[2] = {128, (uint64_t)n_atoms * 4}, strides[1] = {128};
  uint32_t box[2] = {128, 4};
  return x_make_map(m, ptr, 2, dims, strides, box, false);
}

template <int KIND>
cudaError_t x_set_attr() {
  static std::once_flag once;
  static cudaError_t err = cudaSuccess;
  std::call_once(once, [] {
    err = cudaFuncSetAttribute(mx_gemm_kernel<KIND>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               (int)XCfg<KIND>::smem);
    if (err == cudaSuccess)
      err = cudaFuncSetAttribute(mx_gemm_kernel<KIND>,
                                 cudaFuncAttributeNonPortableClusterSizeAllowed, 0);
  });
  return err;
}

// Clusters of two that can be resident at once (0 if none).
template <int KIND>
int x_pair_clusters(int num_sms) {
  static std::once_flag once;
  static int n = 0;
  std::call_once(once, [num_sms] {
    if (x_set_attr<KIND>() != cudaSuccess) return;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(num_sms & ~1), 1, 1);
    cfg.blockDim = dim3(XTHREADS, 1, 1);
    cfg.dynamicSmemBytes = XCfg<KIND>::smem;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = 2;
    at[0].val.clusterDim.y = 1;
    at[0].val.clusterDim.z = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    int c = 0;
    if (cudaOccupancyMaxActiveClusters(&c, mx_gemm_kernel<KIND>, &cfg) == cudaSuccess) n = c;
    else cudaGetLastError();
  });
  return n;
}

template <int KIND>
cudaError_t x_launch(const CUtensorMap& a, const CUtensorMap& b, const CUtensorMap& sa,
                     const CUtensorMap& sb, const XParams& p, int sms, cudaStream_t s) {
  cudaError_t err = x_set_attr<KIND>();
  if (err != cudaSuccess) return err;
  const int clusters = std::min(x_pair_clusters<KIND>(sms), sms / 2);
  if (clusters <= 0) return cudaErrorLaunchOutOfResources;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(2 * clusters), 1, 1);
  cfg.blockDim = dim3(XTHREADS, 1, 1);
  cfg.dynamicSmemBytes = XCfg<KIND>::smem;
  cfg.stream = s;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = 2;
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, mx_gemm_kernel<KIND>, a, b, sa, sb, p);
}

}  // namespace

cudaError_t launch_mx_gemm(const MxGemmCall& g, cudaStream_t s) {
  DeviceInfo di;
  if (device_info(&di) != MOE_OK) return cudaErrorUnknown;
  XParams p{};
  p.row_offsets = g.row_offsets;
  p.dense_rows = g.dense_rows;
  p.row_limit = g.row_offsets ? g.rows : g.dense_rows;
  p.E = g.E;
  p.H = g.H;
  p.d = g.d;
  p.hq = g.hq;
  p.hs = g.hs;
  p.hb = static_cast<bf16*>(g.hb);
  p.abo = static_cast<__half*>(g.abo);
  p.out = g.out;
  p.out_bf16 = g.out_bf16;
  p.abi = static_cast<const __half*>(g.abi);
  p.dgu = static_cast<bf16*>(g.dgu);
  p.dgq = g.dgq;
  p.dgs = g.dgs;
  p.status = g.status;
  CUtensorMap ta, tb, tsa, tsb;
  const uint64_t rows = (uint64_t)g.rows;
  int K;
  bool ok;
  if (g.gate_up) {
    // A: x codes [rows][d]; B: W_gu codes [E][2][H][d] -> dims {d, H, 2, E}
    K = g.d;
    p.n_tiles = g.H / (XBN / 2);
    p.nbt = 2 * g.H / 128;
    uint64_t da[2] = {(uint64_t)g.d, rows}, sa[1] = {(uint64_t)g.d};
    uint32_t ba[2] = {XBK, XBM};
    uint64_t db[4] = {(uint64_t)g.d, (uint64_t)g.H, 2, (uint64_t)g.E};
    uint64_t sb[3] = {(uint64_t)g.d, (uint64_t)g.H * g.d, (uint64_t)2 * g.H * g.d};
    uint32_t bb[4] = {XBK, XBN / 2, 1, 1};
    ok = x_make_map(&ta, g.A, 2, da, sa, ba, true) && x_make_map(&tb, g.B, 4, db, sb, bb, true);
  } else if (g.dh) {
    // A: d_out codes [rows][d]; B: W_down^T codes [E][H][d] -> dims {d, H, E};
    // the output is H wide (the last tile's second half may lie past it)
    K = g.d;
    p.n_tiles = (g.H + XBN - 1) / XBN;
    p.nbt = g.H / 128;
    uint64_t da[2] = {(uint64_t)g.d, rows}, sa[1] = {(uint64_t)g.d};
    uint32_t ba[2] = {XBK, XBM};
    uint64_t db[3] = {(uint64_t)g.d, (uint64_t)g.H, (uint64_t)g.E};
    uint64_t sb[2] = {(uint64_t)g.d, (uint64_t)g.H * g.d};
    uint32_t bb[3] = {XBK, XBN / 2, 1};
    ok = x_make_map(&ta, g.A, 2, da, sa, ba, true) && x_make_map(&tb, g.B, 3, db, sb, bb, true);
  } else {
    // A: h codes [rows][H]; B: W_down codes [E][d][H] -> dims {H, d, E}
    K = g.H;
    p.n_tiles = g.d / XBN;
    p.nbt = g.d / 128;
    uint64_t da[2] = {(uint64_t)g.H, rows}, sa[1] = {(uint64_t)g.H};
    uint32_t ba[2] = {XBK, XBM};
    uint64_t db[3] = {(uint64_t)g.H, (uint64_t)g.d, (uint64_t)g.E};
    uint64_t sb[2] = {(uint64_t)g.H, (uint64_t)g.d * g.H};
    uint32_t bb[3] = {XBK, XBN / 2, 1};
    ok = x_make_map(&ta, g.A, 2, da, sa, ba, true) && x_make_map(&tb, g.B, 3, db, sb, bb, true);
  }
  p.kg = K / XBK;
  ok = ok && x_atom_map(&tsa, g.sfa, (size_t)(rows / XBM) * p.kg) &&
       x_atom_map(&tsb, g.sfb, (size_t)g.E * p.nbt * p.kg);
  if (!ok) return cudaErrorInvalidValue;
  if (g.gate_up && g.hb) return x_launch<MXK_GATE_UP_SAVE>(ta, tb, tsa, tsb, p, di.num_sms, s);
  if (g.gate_up) return x_launch<MXK_GATE_UP>(ta, tb, tsa, tsb, p, di.num_sms, s);
  if (g.dh) return x_launch<MXK_DH>(ta, tb, tsa, tsb, p, di.num_sms, s);
  return x_launch<MXK_DOWN>(ta, tb, tsa, tsb, p, di.num_sms, s);
}

cudaError_t launch_mx_quant_cols(const void* W, uint8_t* Wq, uint8_t* Ws, int groups, int R, int C,
                                 cudaStream_t s) {
  DeviceInfo di;
  if (device_info(&di) != MOE_OK) return cudaErrorUnknown;
  mx_quant_cols_kernel<<<di.num_sms * 8, 256, 0, s>>>(static_cast<const bf16*>(W), Wq, Ws, groups,
                                                      R, C);
  return cudaGetLastError();
}

cudaError_t launch_mx_quant_rows(const void* W, uint8_t* Wq, uint8_t* Ws, long long rows,
                                 long long rows_real, int K, int rows_per_group,
                                 const uint8_t* valid, cudaStream_t s) {
  DeviceInfo di;
  if (device_info(&di) != MOE_OK) return cudaErrorUnknown;
  mx_quant_rows_kernel<<<di.num_sms * 8, 256, 0, s>>>(static_cast<const bf16*>(W), Wq, Ws, rows,
                                                      rows_real, K, rows_per_group, valid);
  return cudaGetLastError();
}

}  // namespace moe
