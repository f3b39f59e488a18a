// Persistent grouped GEMMs of the MoE experts on the 5th-generation tensor
// cores (sm_103a): TMA (cp.async.bulk.tensor, 128-byte swizzle) feeds a
// shared-memory stage ring; one thread issues tcgen05.mma (bf16 x bf16 ->
// fp32) into a double-buffered TMEM accumulator; eight epilogue warps read the
// accumulator back with tcgen05.ld, apply the fused epilogue and store through
// TMA.  By default CTAs work in pairs (cta_group::2): a pair computes a
// 256 x 256 tile, each CTA holding half of A and half of B, which halves the
// B traffic per SM and leaves room for six 32 KB stages.
//
// "spark-gpt" README, Hard-won facts: the MoE experts run as grouped GEMMs
// with the SwiGLU fused into the epilogue (there on GB10 with Triton; here a
// tcgen05/TMEM design for GB300).  "KochiLLM v1.0" card, Configuration: SwiGLU
// experts.
//
// One kernel template covers the five products of the layer:
//   GK_GATE_UP  rows x W_gu[e]^T  -> h = silu(a) * b   (A, B K-major)
//   GK_DOWN     h x W_down[e]^T   -> out               (A, B K-major)
//   GK_DH       d_out x W_down[e] -> SwiGLU backward   (A K-major, B MN-major)
//   GK_DX       d_gu x W_gu[e]    -> dx_perm           (A K-major, B MN-major)
//   GK_DW       A_e^T B_e over the rows of expert e    (A, B MN-major)
// Row-grouped kinds read the expert of each 128-row block from the padded
// segment offsets on the device, so no host synchronisation is needed.
#include <algorithm>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "moe_common.cuh"
#include "moe_internal.h"

namespace moe {

namespace {

constexpr int BM = 128;                  // tile rows per CTA (UMMA M of one CTA)
constexpr int BN = 256;                  // tile columns (UMMA N)
constexpr int BK = 64;                   // K per stage = one 128-byte swizzle row
constexpr int UK = 16;                   // K per tcgen05.mma (bf16)
constexpr int A_BYTES = BM * BK * 2;     // 16 KB
constexpr int TMEM_COLS = 512;           // two 128 x 256 fp32 accumulators
constexpr int THREADS = 384;             // warp 0 TMA, 1 MMA, 2 TMEM, 3 scan, 4-11 epilogue
constexpr int EPI_THREADS = 256;         // two warpgroups split each tile's columns
constexpr int EPI_WARP0 = 4;
constexpr uint64_t WAIT_NS = 2000000000ull;  // bounded waits give up after 2 s
constexpr uint64_t DRAIN_NS = 200000000ull;
constexpr int SLAB_BYTES = 32 * 128;     // per epilogue warp: 32 rows x 128 bytes
constexpr int EPI_WARPS = EPI_THREADS / 32;
constexpr int MAX_STAGES = 6;
// Shared memory: bookkeeping (struct Shared) from the start of the dynamic
// region, the stage ring from the next 1024-byte boundary (128-byte swizzle
// atoms), then the epilogue slabs; 227 KB in all.
constexpr size_t SMEM_BYTES = 232448;
constexpr size_t SHARED_RESERVE = 3072;

// Geometry per product and CTA-group size.  CG = 1: one CTA computes a
// 128 x 256 tile and holds all of B.  CG = 2: a CTA pair computes a 256 x 256
// tile, each CTA holding its 128 rows of A and half of B (128 of the 256
// columns), so a stage is 32 KB and six stages fit.  GK_DH gives one stage up
// for a 4 KB buffer per epilogue warp into which TMA loads the saved a and b
// of the warp's next 32-column chunk.
constexpr int AB_BYTES = 2 * 32 * 64;    // a and b boxes: 32 rows x 32 bf16 each
template <int KIND, int CG>
struct Geo {
  static constexpr int AB_BUF = KIND == GK_DH ? EPI_WARPS * AB_BYTES : 0;
  static constexpr int STAGES = (CG == 2 ? 6 : 4) - (KIND == GK_DH ? 1 : 0);
  static constexpr int B_BYTES = (BN / CG) * BK * 2;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr int RING_BYTES = STAGES * STAGE_BYTES;
  static_assert(SHARED_RESERVE + RING_BYTES + (size_t)EPI_WARPS * SLAB_BYTES + AB_BUF <=
                    SMEM_BYTES,
                "shared memory layout exceeds 227 KB");
};

struct Params {
  const int32_t* row_offsets;  // routed: [E+1] padded offsets; dense: NULL
  int E;
  int rows;                    // dense row count (GK_DW: K rows)
  int K;
  int N;
  int H;
  int Mdw;
  int n_tiles;
  int m_tiles_dw;
  int a_mod;                   // A's K (GK_DOWN) or row (GK_DW) coordinate is taken mod a_mod
  void* out0;        // bf16, or fp32 when out_f32 (GK_DOWN, GK_DX)
  int ld0;
  int out_f32;
  bf16* out1;
  int ld1;
  const bf16* aux_in;
  int ld_aux;
  const uint8_t* valid;
  int* status;
  // GK_DOWN with the combine folded in (dense rows = tokens): y[t] =
  // bf16(sum_j g[t][j] comb_src[comb_inv[t][j]] + acc) into out0 (bf16)
  const bf16* comb_src;        // per-slot rows [R][N] in bf16
  const int32_t* comb_inv;
  const float* comb_gates;
  int comb_k;
  int comb_rows;               // rows of comb_src (debug bounds checks)
  // GK_DX with the dx gather folded in (dense rows = tokens): dx[t] =
  // bf16(sum_j comb_src[comb_inv[t][j]] + acc + router term) into out0; the
  // router term is sum_e dl[t][e] wr[c][e] (rE > 0) or dxr[t][c]
  const float* dl;
  const float* wr;
  int rE;
  const float* dxr;
  // GK_GATE_UP with the permute folded into the A load: row r of the padded
  // permuted layout is token gperm[r] / gk of x (tmA maps x with one-row
  // boxes); pad rows (gperm < 0, or r >= grows) read row gT, past the end,
  // which the TMA fills with zeros
  const int32_t* gperm;
  int gk;
  int gT;
  int grows;
};

struct Shared {
  uint64_t full[MAX_STAGES];
  uint64_t empty[MAX_STAGES];
  uint64_t tfull[2];
  uint64_t tempty[2];
  uint64_t drain;
  uint64_t abfull[EPI_WARPS];  // GK_DH: a|b chunk of each epilogue warp landed
  uint32_t tmem_base;
  int abort_flag;
  int roff[257];               // padded segment offsets (row-grouped kinds)
  int roff_bad;                // debug builds: the segment table failed its check
  int ppre[257];               // CTA pairs: 256-row tiles before expert e (GK_DW: expert order)
};
static_assert(sizeof(Shared) <= SHARED_RESERVE, "bookkeeping too large");

struct Tile {
  int e, m0, n0, kbeg, ksteps, row_end;
};

template <int KIND>
struct KindTraits {
  static constexpr int a_mn = (KIND == GK_DW) ? 1 : 0;
  static constexpr int b_mn = (KIND == GK_DH || KIND == GK_DX || KIND == GK_DW) ? 1 : 0;
  // output columns covered by one tile
  static constexpr int tile_cols = (KIND == GK_GATE_UP) ? BN / 2 : BN;
};

// Last index i in [0, n) with a[i] <= v (a non-decreasing, a[0] <= v).
__device__ __forceinline__ int last_le(const int* a, int n, int v) {
  int lo = 0, hi = n - 1;
  while (lo < hi) {
    int mid = (lo + hi + 1) >> 1;
    if (a[mid] <= v) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// Tiles of one launch.  A tile spans CG * 128 rows: for row-grouped kinds
// with CG = 2 the 128-row blocks of each expert's padded segment are paired
// (an odd last block is paired with rows past the segment, which are computed
// and not stored), so ppre[] counts the pairs before each expert.
template <int KIND, int CG>
__device__ __forceinline__ int num_tiles(const Params& p, const Shared& sh) {
  if (kDebugBounds && p.row_offsets && sh.roff_bad) return 0;
  if (KIND == GK_DW) return p.E * ((p.Mdw + BM * CG - 1) / (BM * CG)) * p.n_tiles;
  int units;
  if (!p.row_offsets) units = (p.rows + BM * CG - 1) / (BM * CG);
  else units = CG == 1 ? sh.roff[p.E] / BM : sh.ppre[p.E];
  return units * p.n_tiles;
}

// Tile idx; m0 is the first row of the tile (the CTA of rank r owns rows
// m0 + 128 r ..), row_end the end of the rows the tile may store.
template <int KIND, int CG>
__device__ __forceinline__ Tile get_tile(const Params& p, const Shared& sh, int idx) {
  Tile t;
  if (KIND == GK_DW) {
    const int m_units = (p.Mdw + BM * CG - 1) / (BM * CG);
    const int per_e = m_units * p.n_tiles;
    const int pos = idx / per_e;                  // position in the heaviest-first order
    t.e = p.row_offsets ? sh.ppre[pos] : pos;
    const int r = idx - pos * per_e;
    t.m0 = (r / p.n_tiles) * BM * CG;
    t.n0 = (r % p.n_tiles) * BN;
    int k0, k1;
    if (p.row_offsets) { k0 = sh.roff[t.e]; k1 = sh.roff[t.e + 1]; }
    else { k0 = 0; k1 = p.rows; }
    t.kbeg = k0;
    t.ksteps = (k1 - k0 + BK - 1) / BK;
    t.row_end = p.Mdw;
  } else {
    const int mu = idx / p.n_tiles;
    t.n0 = (idx - mu * p.n_tiles) * KindTraits<KIND>::tile_cols;
    if (!p.row_offsets) {
      t.e = 0;
      t.m0 = mu * BM * CG;
      t.row_end = p.rows;
    } else if (CG == 1) {
      t.m0 = mu * BM;
      t.e = last_le(sh.roff, p.E, t.m0);
      t.row_end = sh.roff[t.e + 1];
    } else {
      t.e = last_le(sh.ppre, p.E, mu);
      t.m0 = sh.roff[t.e] + (mu - sh.ppre[t.e]) * BM * 2;
      t.row_end = sh.roff[t.e + 1];
    }
    t.kbeg = 0;
    t.ksteps = (p.K + BK - 1) / BK;
  }
  return t;
}

__device__ __forceinline__ void fail(Shared& sh, int* status) {
  set_status(status, MOE_ERR_TIMEOUT);
  *(volatile int*)&sh.abort_flag = 1;
}

// ------------------------------------------------------------------ producer
// The loads of one stage for this CTA: its 128 rows of A (t.m0 is already
// this CTA's first row) and its share of B (all 256 columns for CG = 1, the
// half `rank` for CG = 2), completing on mbarrier `bar` (a cluster address).
template <int KIND, int CG>
__device__ __forceinline__ void tma_2d(uint32_t dst, const CUtensorMap* m, uint32_t bar, int x,
                                       int y) {
  if (CG == 2) tma_load_2d_pair(dst, m, bar, x, y);
  else tma_load_2d(dst, m, bar, x, y);
}
template <int KIND, int CG>
__device__ __forceinline__ void tma_3d(uint32_t dst, const CUtensorMap* m, uint32_t bar, int x,
                                       int y, int z) {
  if (CG == 2) tma_load_3d_pair(dst, m, bar, x, y, z);
  else tma_load_3d(dst, m, bar, x, y, z);
}
// Four rows of a one-row-box 2D tensor map (tile::gather4): rows y0..y3,
// columns x .. x + box - 1, written as consecutive rows at dst.
template <int CG>
__device__ __forceinline__ void tma_gather4(uint32_t dst, const CUtensorMap* m, uint32_t bar,
                                            int x, int y0, int y1, int y2, int y3) {
  if (CG == 2)
    asm volatile(
        "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.tile::gather4"
        ".mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4, %5, %6}], [%7];"
        :: "r"(dst), "l"(reinterpret_cast<uint64_t>(m)), "r"(x), "r"(y0), "r"(y1), "r"(y2),
           "r"(y3), "r"(bar)
        : "memory");
  else
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile::gather4"
        ".mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4, %5, %6}], [%7];"
        :: "r"(dst), "l"(reinterpret_cast<uint64_t>(m)), "r"(x), "r"(y0), "r"(y1), "r"(y2),
           "r"(y3), "r"(bar)
        : "memory");
}

template <int KIND, int CG>
__device__ __forceinline__ void issue_loads(const Tile& t, int kb, uint32_t sa, uint32_t sb,
                                            uint32_t bar, const CUtensorMap* tmA,
                                            const CUtensorMap* tmB, int a_mod, int rank) {
  const int k0 = t.kbeg + kb * BK;
  const int ka = a_mod ? k0 % a_mod : k0;   // A coordinate along K (repeated A)
  constexpr int BH = BN / CG;               // B columns held by this CTA
  const int nb = t.n0 + BH * rank;          // first B column of this CTA
  if (KIND == GK_GATE_UP) {
    tma_2d<KIND, CG>(sa, tmA, bar, k0, t.m0);
    // gate rows then up rows of the same 128 hidden units
    if (CG == 2) {
      tma_load_4d_pair(sb, tmB, bar, k0, t.n0, rank, t.e);
    } else {
      tma_load_4d(sb, tmB, bar, k0, t.n0, 0, t.e);
      tma_load_4d(sb + Geo<KIND, CG>::B_BYTES / 2, tmB, bar, k0, t.n0, 1, t.e);
    }
  } else if (KIND == GK_DOWN) {
    tma_2d<KIND, CG>(sa, tmA, bar, ka, t.m0);
#pragma unroll
    for (int i = 0; i < BH / 128; ++i)
      tma_3d<KIND, CG>(sb + i * 16384, tmB, bar, k0, nb + 128 * i, t.e);
  } else if (KIND == GK_DH || KIND == GK_DX) {
    tma_2d<KIND, CG>(sa, tmA, bar, k0, t.m0);
#pragma unroll
    for (int i = 0; i < BH / 64; ++i)
      tma_3d<KIND, CG>(sb + i * 8192, tmB, bar, nb + 64 * i, k0, t.e);
  } else {  // GK_DW
#pragma unroll
    for (int i = 0; i < 2; ++i) tma_2d<KIND, CG>(sa + i * 8192, tmA, bar, t.m0 + 64 * i, ka);
#pragma unroll
    for (int i = 0; i < BH / 64; ++i) tma_2d<KIND, CG>(sb + i * 8192, tmB, bar, nb + 64 * i, k0);
  }
}

// ------------------------------------------------------------------ epilogue
// The epilogue's results are rounded to bf16 (8 significant bits), so the
// logistic function uses CUDA's fast exponential and approximate division
// (errors of a few fp32 ulp).  For a -> -inf the denominator overflows to
// +inf and the quotient is 0, the limit of both functions.
__device__ __forceinline__ float sigmoid_f(float a) { return __fdividef(1.f, 1.f + __expf(-a)); }
__device__ __forceinline__ float silu_f(float a) { return __fdividef(a, 1.f + __expf(-a)); }

// One epilogue warp's staging slab: 32 rows x 128 bytes in shared memory,
// 128-byte swizzled (16-byte chunk c of row r at chunk position c ^ (r % 8)),
// which is the layout of the output tensor maps' boxes: the warp fills it from
// registers without bank conflicts and one TMA store writes it out as whole
// 128-byte lines.
struct Slab {
  unsigned char* gen;
  uint32_t addr;
};

__device__ __forceinline__ void slab_put(const Slab& s, int lane, int c, const uint4& v) {
  *reinterpret_cast<uint4*>(s.gen + lane * 128 + ((c ^ (lane & 7)) << 4)) = v;
}
// Before the slab is refilled, the previous store must have read it.
__device__ __forceinline__ void slab_acquire(int lane) {
  if (lane == 0) bulk_wait_read0();
  __syncwarp();
}
__device__ __forceinline__ void slab_store(const Slab& s, const CUtensorMap* m, int lane, int x,
                                           int y, int z, bool three_d) {
  fence_proxy_async_smem();
  __syncwarp();
  if (lane == 0) {
    if (three_d) tma_store_3d(m, s.addr, x, y, z);
    else tma_store_2d(m, s.addr, x, y);
    bulk_commit();
  }
}

// GK_DH: the saved pre-activations a and b of one epilogue warp's 32 rows and
// one 32-column chunk, loaded by TMA (two 32 x 32 bf16 boxes in the 64-byte
// swizzle, a then b) into the warp's 4 KB buffer, completing on its mbarrier.
struct AbPipe {
  unsigned char* gen;
  uint32_t addr;
  uint32_t bar;
  uint32_t phase;
  bool pending;
};
__device__ __forceinline__ int ab_col(const Tile& t, int half, int c) {
  return t.n0 + half * 128 + c * 32;
}
__device__ __forceinline__ void ab_issue(AbPipe& ab, const CUtensorMap* tm, const Params& p,
                                         const Tile& t, int row0, int half, int c, int lane) {
  const int col = ab_col(t, half, c);
  if (col >= p.N) return;
  if (lane == 0) {
    mbar_arrive_expect_tx(ab.bar, AB_BYTES);
    tma_load_2d(ab.addr, tm, ab.bar, col, row0);
    tma_load_2d(ab.addr + AB_BYTES / 2, tm, ab.bar, col + p.H, row0);
  }
  ab.pending = true;
}
__device__ __forceinline__ bool ab_wait(AbPipe& ab, volatile int* abort_flag) {
  const bool ok = mbar_wait_bounded(ab.bar, ab.phase, abort_flag, WAIT_NS);
  ab.phase ^= 1u;
  ab.pending = false;
  return ok;
}

// Epilogue of one tile for one warp: TMEM lanes (rows) q*32 .. q*32+31 and
// the column half `half` of the tile (two warpgroups split the columns).
// t.m0 is this CTA's first row.  Rows past the end of the output (dense
// tails, dW rows past M) are clipped by the TMA store; a slab starting at or
// past t.row_end (a segment's end is a multiple of 128 rows) is skipped.
template <int KIND>
__device__ __forceinline__ void epilogue_tile(const Params& p, const Tile& t, uint32_t tacc,
                                              int q, int lane, int half, const Slab& slab,
                                              const CUtensorMap* tmO0, const CUtensorMap* tmO1,
                                              AbPipe& ab, volatile int* abort_flag) {
  const int row0 = t.m0 + q * 32;
  const int row = row0 + lane;
  const int row_end = t.row_end;
  if (row0 >= row_end) return;
  const bool row_in = row < row_end;
  uint32_t r0[32], r1[32];
  if (KIND == GK_GATE_UP) {
    const int col = t.n0 + half * 64;              // 64 hidden units per half
    if (col >= p.H) return;
    const bool zero_row = p.valid && row_in && p.valid[row] == 0;
    slab_acquire(lane);
#pragma unroll 1
    for (int c = 0; c < 2; ++c) {                  // h = silu(a) * b
      const int cb = half * 2 + c;
      __syncwarp();
      tmem_ld32(tacc + cb * 32, r0);
      tmem_ld32(tacc + BN / 2 + cb * 32, r1);
      tmem_ld_wait();
#pragma unroll
      for (int qq = 0; qq < 4; ++qq) {
        float hf[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const float a = zero_row ? 0.f : __uint_as_float(r0[qq * 8 + u]);
          const float b = zero_row ? 0.f : __uint_as_float(r1[qq * 8 + u]);
          hf[u] = silu_f(a) * b;
        }
        slab_put(slab, lane, c * 4 + qq, pack8(hf));
      }
    }
    slab_store(slab, tmO0, lane, col, row0, 0, false);
    if (p.out1) {
#pragma unroll 1
      for (int which = 0; which < 2; ++which) {    // saved a, then b
        slab_acquire(lane);
#pragma unroll 1
        for (int c = 0; c < 2; ++c) {
          __syncwarp();
          tmem_ld32(tacc + which * (BN / 2) + (half * 2 + c) * 32, r0);
          tmem_ld_wait();
#pragma unroll
          for (int qq = 0; qq < 4; ++qq) {
            float v[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) v[u] = zero_row ? 0.f : __uint_as_float(r0[qq * 8 + u]);
            slab_put(slab, lane, c * 4 + qq, pack8(v));
          }
        }
        slab_store(slab, tmO1, lane, col + which * p.H, row0, 0, false);
      }
    }
  } else if (KIND == GK_DH) {
    // dH -> (da, db) with the saved pre-activations a, b, one 32-column chunk
    // at a time: a|b of chunk c arrive by TMA (chunk 0 was issued before the
    // accumulator was waited for; chunk c + 1 is issued once chunk c is in
    // registers); da fills the slab's first half and db its second, each a
    // 32 x 64-byte box in the 64-byte swizzle (16-byte chunk q of row r at
    // q ^ ((r / 2) % 4)), stored to d_gu at columns col and H + col.
    const int swz = (lane >> 1) & 3;
#pragma unroll 1
    for (int c = 0; c < 4; ++c) {
      const int col = ab_col(t, half, c);
      if (col >= p.N) break;
      if (!ab_wait(ab, abort_flag)) {
        if (lane == 0) {
          set_status(p.status, MOE_ERR_TIMEOUT);
          *abort_flag = 1;
        }
        return;
      }
      uint4 av[4], bv[4];
#pragma unroll
      for (int qq = 0; qq < 4; ++qq) {
        const int pos = ((qq ^ swz) << 4) + lane * 64;
        av[qq] = *reinterpret_cast<const uint4*>(ab.gen + pos);
        bv[qq] = *reinterpret_cast<const uint4*>(ab.gen + AB_BYTES / 2 + pos);
      }
      __syncwarp();
      if (c + 1 < 4) ab_issue(ab, tmO1, p, t, row0, half, c + 1, lane);
      __syncwarp();
      tmem_ld32(tacc + (half * 4 + c) * 32, r0);
      tmem_ld_wait();
      slab_acquire(lane);
#pragma unroll
      for (int qq = 0; qq < 4; ++qq) {
        float a8[8], b8[8], da[8], db[8];
        unpack8(av[qq], a8);
        unpack8(bv[qq], b8);
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const float dh = __uint_as_float(r0[qq * 8 + u]);
          const float a = a8[u], b = b8[u];
          const float sg = sigmoid_f(a);
          da[u] = dh * b * sg * (1.f + a * (1.f - sg));
          db[u] = dh * (a * sg);
        }
        const int pos = (qq ^ swz) << 4;
        *reinterpret_cast<uint4*>(slab.gen + lane * 64 + pos) = pack8(da);
        *reinterpret_cast<uint4*>(slab.gen + 2048 + lane * 64 + pos) = pack8(db);
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        tma_store_2d(tmO0, slab.addr, col, row0);
        tma_store_2d(tmO0, slab.addr + 2048, col + p.H, row0);
        bulk_commit();
      }
    }
  } else {
    // GK_DOWN, GK_DX, GK_DW: 128 columns per half
    const bool no_acc = t.ksteps == 0;
    const bool three_d = KIND == GK_DW;
    if (KIND == GK_DOWN && p.comb_src) {
      // the combine, for token t = row: y = sum_j g_j out_perm[inv(t, j)]
      // (fp32, slot order, unused slots skipped) + this GEMM's value, one
      // rounding to bf16 -- the combine kernel's operations in its order;
      // PAD tokens get 0
      const bool real = row_in && (p.valid == nullptr || p.valid[row] != 0);
      const int32_t* inv_t = p.comb_inv + (size_t)row * p.comb_k;
      const float* g_t = p.comb_gates + (size_t)row * p.comb_k;
#pragma unroll 1
      for (int bx = 0; bx < 2; ++bx) {             // one 64-column bf16 box per two chunks
        const int col = t.n0 + half * 128 + bx * 64;
        if (col >= p.N) break;
        slab_acquire(lane);
#pragma unroll 1
        for (int c = 0; c < 2; ++c) {
          float acc[32];
#pragma unroll
          for (int u = 0; u < 32; ++u) acc[u] = 0.f;
          if (real) {
            for (int j = 0; j < p.comb_k; ++j) {
              const int r = dbg_row(inv_t[j], p.comb_rows, p.status);
              if (r < 0) continue;
              const float g = g_t[j];
              const bf16* src = p.comb_src + (size_t)r * p.N + col + c * 32;
#pragma unroll
              for (int i = 0; i < 4; ++i) {
                float v[8];
                unpack8(ld_nc_v4(src + i * 8), v);
#pragma unroll
                for (int u = 0; u < 8; ++u) acc[i * 8 + u] = fmaf(g, v[u], acc[i * 8 + u]);
              }
            }
          }
          __syncwarp();
          tmem_ld32(tacc + (half * 4 + bx * 2 + c) * 32, r0);
          tmem_ld_wait();
#pragma unroll
          for (int u = 0; u < 32; ++u)
            acc[u] = real ? acc[u] + __uint_as_float(r0[u]) : 0.f;
#pragma unroll
          for (int qq = 0; qq < 4; ++qq) slab_put(slab, lane, c * 4 + qq, pack8(&acc[qq * 8]));
        }
        slab_store(slab, tmO0, lane, col, row0, 0, false);
      }
    } else if (KIND == GK_DX && p.comb_src) {
      // the dx gather, for token t = row: dx = sum_j dx_perm[inv(t, j)]
      // (slot order, unused slots skipped) + this GEMM's value + the router
      // term, one rounding to bf16 -- the gather kernel's operations in its
      // order; PAD tokens get 0
      const bool real = row_in && (p.valid == nullptr || p.valid[row] != 0);
      const int32_t* inv_t = p.comb_inv + (size_t)row * p.comb_k;
      const float4* dl_t = reinterpret_cast<const float4*>(p.dl + (size_t)row * p.rE);
#pragma unroll 1
      for (int bx = 0; bx < 2; ++bx) {             // one 64-column bf16 box per two chunks
        const int col = t.n0 + half * 128 + bx * 64;
        if (col >= p.N) break;
        slab_acquire(lane);
#pragma unroll 1
        for (int c = 0; c < 4; ++c) {              // 16 columns at a time
          const int c0 = col + c * 16;
          float acc[16];
#pragma unroll
          for (int u = 0; u < 16; ++u) acc[u] = 0.f;
          if (real) {
            for (int j = 0; j < p.comb_k; ++j) {
              const int r = dbg_row(inv_t[j], p.comb_rows, p.status);
              if (r < 0) continue;
              const bf16* src = p.comb_src + (size_t)r * p.N + c0;
#pragma unroll
              for (int i = 0; i < 2; ++i) {
                float v[8];
                unpack8(ld_nc_v4(src + i * 8), v);
#pragma unroll
                for (int u = 0; u < 8; ++u) acc[i * 8 + u] += v[u];
              }
            }
          }
          uint32_t r16[16];
          __syncwarp();
          tmem_ld16(tacc + (half * 4 + bx * 2) * 32 + c * 16, r16);
          tmem_ld_wait();
          if (real) {
#pragma unroll
            for (int u = 0; u < 16; ++u) acc[u] += __uint_as_float(r16[u]);
            if (p.rE > 0) {
              // sum_e dl[t][e] W_r[c][e] per column c, e in order (experts
              // outside, columns inside: 16 running sums, 4 coefficients live)
              float sr[16];
#pragma unroll
              for (int u = 0; u < 16; ++u) sr[u] = 0.f;
#pragma unroll 1
              for (int e4 = 0; e4 < p.rE; e4 += 4) {
                const float4 dv = __ldg(dl_t + e4 / 4);
#pragma unroll
                for (int u = 0; u < 16; ++u) {
                  const float4 wv =
                      __ldg(reinterpret_cast<const float4*>(p.wr + (size_t)(c0 + u) * p.rE + e4));
                  sr[u] = fmaf(dv.x, wv.x, sr[u]);
                  sr[u] = fmaf(dv.y, wv.y, sr[u]);
                  sr[u] = fmaf(dv.z, wv.z, sr[u]);
                  sr[u] = fmaf(dv.w, wv.w, sr[u]);
                }
              }
#pragma unroll
              for (int u = 0; u < 16; ++u) acc[u] += sr[u];
            } else if (p.dxr) {
              const float* pr = p.dxr + (size_t)row * p.N + c0;
#pragma unroll
              for (int i = 0; i < 4; ++i) {
                const uint4 v = ld_nc_v4(pr + i * 4);
                acc[i * 4 + 0] += __uint_as_float(v.x);
                acc[i * 4 + 1] += __uint_as_float(v.y);
                acc[i * 4 + 2] += __uint_as_float(v.z);
                acc[i * 4 + 3] += __uint_as_float(v.w);
              }
            }
          } else {
#pragma unroll
            for (int u = 0; u < 16; ++u) acc[u] = 0.f;
          }
          slab_put(slab, lane, c * 2, pack8(&acc[0]));
          slab_put(slab, lane, c * 2 + 1, pack8(&acc[8]));
        }
        slab_store(slab, tmO0, lane, col, row0, 0, false);
      }
    } else if (p.out_f32) {
#pragma unroll 1
      for (int c = 0; c < 4; ++c) {                // one 32-column fp32 box per chunk
        const int col = t.n0 + half * 128 + c * 32;
        if (col >= p.N) break;
        slab_acquire(lane);
        __syncwarp();
        tmem_ld32(tacc + (half * 4 + c) * 32, r0);
        tmem_ld_wait();
#pragma unroll
        for (int qq = 0; qq < 8; ++qq)
          slab_put(slab, lane, qq,
                   no_acc ? make_uint4(0, 0, 0, 0)
                          : make_uint4(r0[qq * 4], r0[qq * 4 + 1], r0[qq * 4 + 2], r0[qq * 4 + 3]));
        slab_store(slab, tmO0, lane, col, row0, t.e, three_d);
      }
    } else {
#pragma unroll 1
      for (int bx = 0; bx < 2; ++bx) {             // one 64-column bf16 box per two chunks
        const int col = t.n0 + half * 128 + bx * 64;
        if (col >= p.N) break;
        slab_acquire(lane);
#pragma unroll 1
        for (int c = 0; c < 2; ++c) {
          __syncwarp();
          tmem_ld32(tacc + (half * 4 + bx * 2 + c) * 32, r0);
          tmem_ld_wait();
#pragma unroll
          for (int qq = 0; qq < 4; ++qq) {
            float v[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) v[u] = no_acc ? 0.f : __uint_as_float(r0[qq * 8 + u]);
            slab_put(slab, lane, c * 4 + qq, pack8(v));
          }
        }
        slab_store(slab, tmO0, lane, col, row0, t.e, three_d);
      }
    }
  }
}

// ------------------------------------------------------------------ kernel
// CG = 1: every CTA works alone.  CG = 2: CTAs run in clusters of two; the
// even CTA (rank 0) issues the pair MMAs, both load their shares of each
// stage (completing on rank 0's full barrier), the MMA commits arrive on both
// CTAs' empty and accumulator-full barriers, and both CTAs' epilogue warps
// arrive on rank 0's accumulator-empty barrier.
template <int KIND, int CG>
__global__ void __launch_bounds__(THREADS, 1)
grouped_gemm_kernel(const __grid_constant__ CUtensorMap tmA,
                    const __grid_constant__ CUtensorMap tmB,
                    const __grid_constant__ CUtensorMap tmO0,
                    const __grid_constant__ CUtensorMap tmO1, const Params p) {
  using G = Geo<KIND, CG>;
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + (uint32_t)sizeof(Shared) + 1023u) & ~1023u;
  // the layout must fit the allocation (it does whenever the dynamic region
  // starts 1024-byte aligned); both CTAs of a pair see the same addresses,
  // so both return here together
  if (base - raw + (size_t)G::RING_BYTES + (size_t)EPI_WARPS * SLAB_BYTES + G::AB_BUF >
      SMEM_BYTES) {
    if (threadIdx.x == 0) set_status(p.status, MOE_ERR_DEVICE);
    return;
  }
  Shared& sh = *reinterpret_cast<Shared*>(smem_raw);
  unsigned char* slabs = smem_raw + (base - raw) + (size_t)G::RING_BYTES;
  unsigned char* abbuf = slabs + (size_t)EPI_WARPS * SLAB_BYTES;   // GK_DH only

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int rank = CG == 2 ? (int)cluster_ctarank() : 0;
  const int unit = CG == 2 ? (int)(blockIdx.x >> 1) : (int)blockIdx.x;   // cluster index
  const int nunits = CG == 2 ? (int)(gridDim.x >> 1) : (int)gridDim.x;

  if (threadIdx.x == 0) {
    for (int s = 0; s < G::STAGES; ++s) {
      mbar_init(smem_u32(&sh.full[s]), 1);
      mbar_init(smem_u32(&sh.empty[s]), 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(smem_u32(&sh.tfull[a]), 1);
      mbar_init(smem_u32(&sh.tempty[a]), CG == 2 ? 2 * EPI_WARPS : EPI_THREADS);
    }
    mbar_init(smem_u32(&sh.drain), 1);
    for (int w = 0; w < EPI_WARPS; ++w) mbar_init(smem_u32(&sh.abfull[w]), 1);
    sh.abort_flag = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
    tma_prefetch_desc(&tmO0);
    if (p.out1 || KIND == GK_DH) tma_prefetch_desc(&tmO1);
  }
  if (p.row_offsets)
    for (int e = threadIdx.x; e <= p.E; e += blockDim.x) sh.roff[e] = p.row_offsets[e];
  if (warp == 2) {
    if (CG == 2) {
      tmem_alloc_pair(smem_u32(&sh.tmem_base), TMEM_COLS);
      tmem_relinquish_pair();
    } else {
      tmem_alloc(smem_u32(&sh.tmem_base), TMEM_COLS);
      tmem_relinquish();
    }
  }
  tc_fence_before();
  __syncthreads();
  if (kDebugBounds && p.row_offsets && threadIdx.x == 0) {
    sh.roff_bad = dbg_roff_ok(sh.roff, p.E, p.rows) ? 0 : 1;
    if (sh.roff_bad) set_status(p.status, MOE_ERR_BOUNDS);
  }
  if (CG == 2 && KIND != GK_DW && p.row_offsets && warp == 3) {
    // 256-row tiles per expert (pairs of 128-row blocks), prefix over experts
    int carry = 0;
    for (int e0 = 0; e0 < p.E; e0 += 32) {
      const int e = e0 + lane;
      int v = e < p.E ? ((sh.roff[e + 1] - sh.roff[e]) / BM + 1) / 2 : 0;
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
  if (KIND == GK_DW && p.row_offsets) {
    // Heaviest experts first: the dW tiles are taken in the order of their
    // expert's segment length (the tile's K), longest first, equal lengths
    // in index order (ppre, unused by this kind, holds that order).  Unit u
    // takes tiles u, u + nunits, ..., so the long K loops of skewed experts
    // are spread over the units first and the short ones fill in behind.
    for (int e = threadIdx.x; e < p.E; e += blockDim.x) {
      const int le = sh.roff[e + 1] - sh.roff[e];
      int r = 0;
      for (int f = 0; f < p.E; ++f) {
        const int lf = sh.roff[f + 1] - sh.roff[f];
        r += (lf > le) || (lf == le && f < e);
      }
      sh.ppre[r] = e;
    }
  }
  // barriers of both CTAs initialised (the pair signals across CTAs)
  if (CG == 2) cluster_sync();
  else __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sh.tmem_base;
  const int ntiles = num_tiles<KIND, CG>(p, sh);
  volatile int* abort_flag = &sh.abort_flag;

  if (warp == 0) {
    // ---------------- TMA producer (both CTAs): lane 0 waits for free stages
    // and issues the box loads; with the permute folded in (GK_GATE_UP,
    // gperm set) every lane also gathers four of the stage's 128 A rows
    const bool gather = KIND == GK_GATE_UP && p.gperm != nullptr;
    int stage = 0;
    uint32_t phase = 0;
    int pending_parity[MAX_STAGES];
    for (int s = 0; s < G::STAGES; ++s) pending_parity[s] = -1;
    bool ok = true;
    for (int idx = unit; idx < ntiles && ok; idx += nunits) {
      Tile t = get_tile<KIND, CG>(p, sh, idx);
      t.m0 += BM * rank;
      int tok[4] = {0, 0, 0, 0};
      if (gather) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int r = t.m0 + lane * 4 + i;
          const int pp = r < p.grows ? p.gperm[r] : -1;
          tok[i] = pp >= 0 ? pp / p.gk : p.gT;
        }
      }
      for (int kb = 0; kb < t.ksteps; ++kb) {
        int good = 1;
        if (lane == 0)
          good = mbar_wait_bounded(smem_u32(&sh.empty[stage]), phase ^ 1u, abort_flag, WAIT_NS);
        good = __shfl_sync(0xffffffffu, good, 0);
        if (!good) {
          if (lane == 0) fail(sh, p.status);
          ok = false;
          break;
        }
        const uint32_t fb_local = smem_u32(&sh.full[stage]);
        // the stage's bytes from both CTAs complete on rank 0's barrier
        const uint32_t fb = CG == 2 ? mapa_shared(fb_local, 0) : fb_local;
        if (lane == 0 && rank == 0) mbar_arrive_expect_tx(fb_local, G::STAGE_BYTES * CG);
        const uint32_t sa = base + stage * G::STAGE_BYTES;
        if (gather) {
          const int k0 = t.kbeg + kb * BK;
          tma_gather4<CG>(sa + lane * 4 * 128, &tmA, fb, k0, tok[0], tok[1], tok[2], tok[3]);
          if (lane == 0) {
            if (CG == 2) {
              tma_load_4d_pair(sa + A_BYTES, &tmB, fb, k0, t.n0, rank, t.e);
            } else {
              tma_load_4d(sa + A_BYTES, &tmB, fb, k0, t.n0, 0, t.e);
              tma_load_4d(sa + A_BYTES + G::B_BYTES / 2, &tmB, fb, k0, t.n0, 1, t.e);
            }
          }
        } else if (lane == 0) {
          issue_loads<KIND, CG>(t, kb, sa, sa + A_BYTES, fb, &tmA, &tmB, p.a_mod, rank);
        }
        pending_parity[stage] = (int)phase;
        if (++stage == G::STAGES) { stage = 0; phase ^= 1u; }
      }
    }
    if (!ok && lane == 0) {
      // let every copy already issued land before shared memory is released
      if (CG == 1) {
        for (int s = 0; s < G::STAGES; ++s)
          if (pending_parity[s] >= 0) {
            int dummy = 0;
            mbar_wait_bounded(smem_u32(&sh.full[s]), (uint32_t)pending_parity[s], &dummy,
                              DRAIN_NS);
          }
      } else {
        // this CTA's copies complete on rank 0's barriers: give them a
        // bounded time instead
        const uint64_t t0 = global_ns();
        while (global_ns() - t0 < DRAIN_NS) {
        }
      }
    }
  } else if (warp == 1 && lane == 0 && rank == 0) {
    // ---------------- MMA issuer (rank 0 of a pair)
    constexpr uint32_t idesc =
        umma_idesc_bf16(BM * CG, BN, KindTraits<KIND>::a_mn, KindTraits<KIND>::b_mn);
    constexpr uint32_t a_step = KindTraits<KIND>::a_mn ? 16 * 128 : UK * 2;
    constexpr uint32_t b_step = KindTraits<KIND>::b_mn ? 16 * 128 : UK * 2;
    constexpr uint32_t a_lbo = KindTraits<KIND>::a_mn ? 8192 : 16;
    constexpr uint32_t b_lbo = KindTraits<KIND>::b_mn ? 8192 : 16;
    int stage = 0;
    uint32_t phase = 0;
    int it = 0;
    bool ok = true;
    for (int idx = unit; idx < ntiles && ok; idx += nunits, ++it) {
      const Tile t = get_tile<KIND, CG>(p, sh, idx);
      const int acc = it & 1;
      const uint32_t acc_phase = (it >> 1) & 1;
      const bool freed =
          CG == 2 ? mbar_wait_bounded_cluster(smem_u32(&sh.tempty[acc]), acc_phase ^ 1u,
                                              abort_flag, WAIT_NS)
                  : mbar_wait_bounded(smem_u32(&sh.tempty[acc]), acc_phase ^ 1u, abort_flag,
                                      WAIT_NS);
      if (!freed) {
        fail(sh, p.status);
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t d_tmem = tmem + acc * BN;
      for (int kb = 0; kb < t.ksteps; ++kb) {
        if (!mbar_wait_bounded(smem_u32(&sh.full[stage]), phase, abort_flag, WAIT_NS)) {
          fail(sh, p.status);
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t sa = base + stage * G::STAGE_BYTES;
        const uint32_t sb = sa + A_BYTES;
#pragma unroll
        for (int kk = 0; kk < BK / UK; ++kk) {
          const uint64_t ad = umma_desc_sw128(sa + kk * a_step, a_lbo, 1024);
          const uint64_t bd = umma_desc_sw128(sb + kk * b_step, b_lbo, 1024);
          if (CG == 2) umma_bf16_pair(d_tmem, ad, bd, idesc, (kb | kk) != 0 ? 1u : 0u);
          else umma_bf16(d_tmem, ad, bd, idesc, (kb | kk) != 0 ? 1u : 0u);
        }
        if (CG == 2) umma_commit_pair(smem_u32(&sh.empty[stage]), 3);
        else umma_commit(smem_u32(&sh.empty[stage]));
        if (++stage == G::STAGES) { stage = 0; phase ^= 1u; }
      }
      if (!ok) break;
      if (CG == 2) umma_commit_pair(smem_u32(&sh.tfull[acc]), 3);
      else umma_commit(smem_u32(&sh.tfull[acc]));
    }
    // all issued MMAs complete before TMEM can be released
    if (CG == 2) umma_commit_pair(smem_u32(&sh.drain), 1);
    else umma_commit(smem_u32(&sh.drain));
    int dummy = 0;
    mbar_wait_bounded(smem_u32(&sh.drain), 0, &dummy, DRAIN_NS);
  } else if (warp >= EPI_WARP0) {
    // ---------------- epilogue warps: TMEM lanes 32*(warp%4) .. +31
    const int q = warp & 3;                       // TMEM lane quadrant of this warp
    const int half = (warp - EPI_WARP0) >> 2;     // column half of the tile
    Slab slab;
    slab.gen = slabs + (size_t)(warp - EPI_WARP0) * SLAB_BYTES;
    slab.addr = smem_u32(slab.gen);
    int it = 0;
    AbPipe ab;
    ab.gen = abbuf + (size_t)(warp - EPI_WARP0) * AB_BYTES;
    ab.addr = smem_u32(ab.gen);
    ab.bar = smem_u32(&sh.abfull[warp - EPI_WARP0]);
    ab.phase = 0;
    ab.pending = false;
    for (int idx = unit; idx < ntiles; idx += nunits, ++it) {
      Tile t = get_tile<KIND, CG>(p, sh, idx);
      t.m0 += BM * rank;
      // a|b of the tile's first chunk, unless this warp's rows are all past
      // the tile's end (then the epilogue skips them)
      if (KIND == GK_DH && t.m0 + q * 32 < t.row_end)
        ab_issue(ab, &tmO1, p, t, t.m0 + q * 32, half, 0, lane);
      const int acc = it & 1;
      const uint32_t acc_phase = (it >> 1) & 1;
      if (!mbar_wait_bounded(smem_u32(&sh.tfull[acc]), acc_phase, abort_flag, WAIT_NS)) {
        if (lane == 0) fail(sh, p.status);
        break;
      }
      tc_fence_after();
      const uint32_t tacc = tmem + ((uint32_t)(q * 32) << 16) + acc * BN;
      epilogue_tile<KIND>(p, t, tacc, q, lane, half, slab, &tmO0, &tmO1, ab, abort_flag);
      tc_fence_before();
      if (CG == 2) {
        __syncwarp();
        if (lane == 0) mbar_arrive_cluster(mapa_shared(smem_u32(&sh.tempty[acc]), 0));
      } else {
        mbar_arrive(smem_u32(&sh.tempty[acc]));
      }
    }
    // a copy still on its way into this warp's a|b buffer lands, and every
    // store issued from its slab completes, before exit
    if (KIND == GK_DH && ab.pending) {
      int dummy = 0;
      mbar_wait_bounded(ab.bar, ab.phase, &dummy, DRAIN_NS);
    }
    if (lane == 0) bulk_wait0();
    __syncwarp();
  }
  __syncwarp();
  tc_fence_before();
  // no CTA of a pair leaves (or frees TMEM) while its peer may still signal
  // its barriers or the pair's MMAs may still write its TMEM
  if (CG == 2) cluster_sync();
  else __syncthreads();
  if (warp == 2) {
    tc_fence_after();
    if (CG == 2) tmem_dealloc_pair(tmem, TMEM_COLS);
    else tmem_dealloc(tmem, TMEM_COLS);
  }
}

// ------------------------------------------------------------------ host side
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                         cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(ptr);
  });
  return fn;
}

// bf16 tensor map, 128-byte swizzle, zero fill out of bounds.
// dims/strides: innermost first; strides in bytes for dims 1..rank-1.
bool make_map(CUtensorMap* m, const void* ptr, int rank, const uint64_t* dims,
              const uint64_t* strides, const uint32_t* box,
              CUtensorMapDataType dtype = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
              CUtensorMapSwizzle swz = CU_TENSOR_MAP_SWIZZLE_128B) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t gd[5], gs[4];
  cuuint32_t bx[5], es[5];
  for (int i = 0; i < rank; ++i) { gd[i] = dims[i]; bx[i] = box[i]; es[i] = 1; }
  for (int i = 0; i < rank - 1; ++i) gs[i] = strides[i];
  CUresult r = fn(m, dtype, (cuuint32_t)rank, const_cast<void*>(ptr),
                  gd, gs, bx, es, CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

template <int KIND, int CG>
cudaError_t set_smem_attr() {
  static std::once_flag once;
  static cudaError_t err = cudaSuccess;
  std::call_once(once, [] {
    err = cudaFuncSetAttribute(grouped_gemm_kernel<KIND, CG>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SMEM_BYTES);
    if (err == cudaSuccess && CG == 2)
      err = cudaFuncSetAttribute(grouped_gemm_kernel<KIND, CG>,
                                 cudaFuncAttributeNonPortableClusterSizeAllowed, 0);
  });
  return err;
}

// Clusters of two that can be resident at once (0 if none), per kind.
template <int KIND>
int pair_clusters(int num_sms) {
  static std::once_flag once;
  static int n = 0;
  std::call_once(once, [num_sms] {
    if (set_smem_attr<KIND, 2>() != cudaSuccess) return;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(num_sms & ~1), 1, 1);
    cfg.blockDim = dim3(THREADS, 1, 1);
    cfg.dynamicSmemBytes = SMEM_BYTES;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = 2;
    at[0].val.clusterDim.y = 1;
    at[0].val.clusterDim.z = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    int c = 0;
    if (cudaOccupancyMaxActiveClusters(&c, grouped_gemm_kernel<KIND, 2>, &cfg) == cudaSuccess)
      n = c;
    else
      cudaGetLastError();
  });
  return n;
}

template <int KIND>
cudaError_t launch_kind(const CUtensorMap& a, const CUtensorMap& b, const CUtensorMap& o0,
                        const CUtensorMap& o1, const Params& p, int num_sms, bool pairs,
                        cudaStream_t s) {
  if (pairs) {
    const int clusters = std::min(pair_clusters<KIND>(num_sms), num_sms / 2);
    if (clusters > 0) {
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3((unsigned)(2 * clusters), 1, 1);
      cfg.blockDim = dim3(THREADS, 1, 1);
      cfg.dynamicSmemBytes = SMEM_BYTES;
      cfg.stream = s;
      cudaLaunchAttribute at[1];
      at[0].id = cudaLaunchAttributeClusterDimension;
      at[0].val.clusterDim.x = 2;
      at[0].val.clusterDim.y = 1;
      at[0].val.clusterDim.z = 1;
      cfg.attrs = at;
      cfg.numAttrs = 1;
      return cudaLaunchKernelEx(&cfg, grouped_gemm_kernel<KIND, 2>, a, b, o0, o1, p);
    }
  }
  cudaError_t err = set_smem_attr<KIND, 1>();
  if (err != cudaSuccess) return err;
  grouped_gemm_kernel<KIND, 1><<<num_sms, THREADS, SMEM_BYTES, s>>>(a, b, o0, o1, p);
  return cudaGetLastError();
}

// Which kernel the products run on: CTA pairs (6-12% faster than single CTAs
// for every product on the KochiLLM and 128-expert shapes, 20% for DH at
// K = 1536), or the single-CTA kernel where a cluster of two cannot be
// launched.  MOE_GEMM_CTA_PAIRS=0 forces single CTAs (for measurement).
bool use_pairs() {
  const char* v = getenv("MOE_GEMM_CTA_PAIRS");
  return !(v && v[0] == '0');
}

}  // namespace

cudaError_t launch_gemm(const GemmCall& g, cudaStream_t s) {
  static_assert(sizeof(Shared) <= SHARED_RESERVE, "shared bookkeeping too large");
  static_assert(SMEM_BYTES <= 232448, "exceeds the 227 KB opt-in shared memory of a block");
  DeviceInfo di;
  if (device_info(&di) != MOE_OK) return cudaErrorUnknown;
  CUtensorMap ta, tb;
  Params p{};
  p.row_offsets = g.row_offsets;
  p.E = g.E;
  p.rows = g.rows;
  p.K = g.K;
  p.N = g.N;
  p.H = g.H;
  p.Mdw = g.Mdw;
  p.out0 = g.out0;
  p.ld0 = g.ld0;
  p.out_f32 = g.out_f32;
  p.a_mod = g.a_mod;
  p.out1 = static_cast<bf16*>(g.out1);
  p.ld1 = g.ld1;
  p.aux_in = static_cast<const bf16*>(g.aux_in);
  p.ld_aux = g.ld_aux;
  p.valid = g.valid;
  p.status = g.status;
  p.comb_src = static_cast<const bf16*>(g.comb_src);
  p.comb_inv = g.comb_inv;
  p.comb_rows = g.comb_rows;
  p.comb_gates = g.comb_gates;
  p.comb_k = g.comb_k;
  p.dl = g.dl;
  p.wr = g.wr;
  p.rE = g.rE;
  p.dxr = g.dxr;
  p.gperm = g.gperm;
  p.gk = g.gk;
  p.gT = g.gT;
  p.grows = g.grows;
  const uint64_t rows = (uint64_t)g.rows;
  bool ok = true;
  switch (g.kind) {
    case GK_GATE_UP: {
      // A: [rows][K] (or, gathered, x [gT][K] with one-row boxes) ;
      // B: W_gu [E][2][H][K] -> dims {K, H, 2, E}
      uint64_t da[2] = {(uint64_t)g.K, g.gperm ? (uint64_t)g.gT : rows},
               sa[1] = {(uint64_t)g.lda * 2};
      uint32_t ba[2] = {64, g.gperm ? 1u : 128u};
      uint64_t db[4] = {(uint64_t)g.K, (uint64_t)g.H, 2, (uint64_t)g.E};
      uint64_t sb[3] = {(uint64_t)g.K * 2, (uint64_t)g.H * g.K * 2, (uint64_t)2 * g.H * g.K * 2};
      uint32_t bb[4] = {64, 128, 1, 1};
      ok = make_map(&ta, g.A, 2, da, sa, ba) && make_map(&tb, g.B, 4, db, sb, bb);
      p.n_tiles = (g.H + BN / 2 - 1) / (BN / 2);
      break;
    }
    case GK_DOWN: {
      // A: [rows][K=H] (or [rows][a_mod], read K/a_mod times) ; B: W_down [E][N=d][K=H]
      // -> dims {K, N, E}
      uint64_t da[2] = {(uint64_t)(g.a_mod ? g.a_mod : g.K), rows},
               sa[1] = {(uint64_t)g.lda * 2};
      uint32_t ba[2] = {64, 128};
      uint64_t db[3] = {(uint64_t)g.K, (uint64_t)g.N, (uint64_t)g.E};
      uint64_t sb[2] = {(uint64_t)g.K * 2, (uint64_t)g.N * g.K * 2};
      uint32_t bb[3] = {64, 128, 1};
      ok = make_map(&ta, g.A, 2, da, sa, ba) && make_map(&tb, g.B, 3, db, sb, bb);
      p.n_tiles = (g.N + BN - 1) / BN;
      break;
    }
    case GK_DH:
    case GK_DX: {
      // A: [rows][K] ; B: [E][K][N] (N contiguous) -> dims {N, K, E}
      uint64_t da[2] = {(uint64_t)g.K, rows}, sa[1] = {(uint64_t)g.lda * 2};
      uint32_t ba[2] = {64, 128};
      uint64_t db[3] = {(uint64_t)g.N, (uint64_t)g.K, (uint64_t)g.E};
      uint64_t sb[2] = {(uint64_t)g.N * 2, (uint64_t)g.K * g.N * 2};
      uint32_t bb[3] = {64, 64, 1};
      ok = make_map(&ta, g.A, 2, da, sa, ba) && make_map(&tb, g.B, 3, db, sb, bb);
      p.n_tiles = (g.N + BN - 1) / BN;
      break;
    }
    case GK_DW: {
      // A: [a_rows][Mdw] (M contiguous; rows read mod a_mod) ; B: [rows][N] (N contiguous)
      uint64_t da[2] = {(uint64_t)g.Mdw, (uint64_t)(g.a_rows ? g.a_rows : g.rows)},
               sa[1] = {(uint64_t)g.lda * 2};
      uint32_t ba[2] = {64, 64};
      uint64_t db[2] = {(uint64_t)g.N, rows}, sb[1] = {(uint64_t)g.N * 2};
      uint32_t bb[2] = {64, 64};
      ok = make_map(&ta, g.A, 2, da, sa, ba) && make_map(&tb, g.B, 2, db, sb, bb);
      p.n_tiles = (g.N + BN - 1) / BN;
      p.m_tiles_dw = (g.Mdw + BM - 1) / BM;
      break;
    }
  }
  if (!ok) return cudaErrorInvalidValue;
  // Output maps: 128-byte swizzled boxes of 128 bytes x 32 rows (one epilogue
  // warp's slab).  Rows and columns past the tensor are clipped by the store.
  CUtensorMap to0, to1;
  memset(&to0, 0, sizeof(to0));
  memset(&to1, 0, sizeof(to1));
  const int es = g.out_f32 ? 4 : 2;
  const CUtensorMapDataType ot =
      g.out_f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  const uint32_t inner = 128 / es;
  switch (g.kind) {
    case GK_GATE_UP: {
      uint64_t d0[2] = {(uint64_t)g.H, rows}, s0[1] = {(uint64_t)g.ld0 * 2};
      uint32_t b0[2] = {64, 32};
      ok = make_map(&to0, g.out0, 2, d0, s0, b0);
      if (ok && g.out1) {
        uint64_t d1[2] = {(uint64_t)2 * g.H, rows}, s1[1] = {(uint64_t)g.ld1 * 2};
        ok = make_map(&to1, g.out1, 2, d1, s1, b0);
      }
      break;
    }
    case GK_DH: {
      uint64_t d0[2] = {(uint64_t)2 * g.H, rows}, s0[1] = {(uint64_t)g.ld0 * 2};
      uint32_t b0[2] = {32, 32};
      ok = make_map(&to0, g.out0, 2, d0, s0, b0, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                    CU_TENSOR_MAP_SWIZZLE_64B);
      // the second map loads the saved a|b (same box and swizzle)
      uint64_t d1[2] = {(uint64_t)2 * g.H, rows}, s1[1] = {(uint64_t)g.ld_aux * 2};
      ok = ok && make_map(&to1, g.aux_in, 2, d1, s1, b0, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                          CU_TENSOR_MAP_SWIZZLE_64B);
      break;
    }
    case GK_DOWN:
    case GK_DX: {
      uint64_t d0[2] = {(uint64_t)g.N, rows}, s0[1] = {(uint64_t)g.ld0 * es};
      uint32_t b0[2] = {inner, 32};
      ok = make_map(&to0, g.out0, 2, d0, s0, b0, ot);
      break;
    }
    case GK_DW: {
      uint64_t d0[3] = {(uint64_t)g.N, (uint64_t)g.Mdw, (uint64_t)g.E};
      uint64_t s0[2] = {(uint64_t)g.ld0 * es, (uint64_t)g.Mdw * g.ld0 * es};
      uint32_t b0[3] = {inner, 32, 1};
      ok = make_map(&to0, g.out0, 3, d0, s0, b0, ot);
      break;
    }
  }
  if (!ok) return cudaErrorInvalidValue;
  const int sms = di.num_sms;
  const bool pairs = use_pairs();
  switch (g.kind) {
    case GK_GATE_UP: return launch_kind<GK_GATE_UP>(ta, tb, to0, to1, p, sms, pairs, s);
    case GK_DOWN: return launch_kind<GK_DOWN>(ta, tb, to0, to1, p, sms, pairs, s);
    case GK_DH: return launch_kind<GK_DH>(ta, tb, to0, to1, p, sms, pairs, s);
    case GK_DX: return launch_kind<GK_DX>(ta, tb, to0, to1, p, sms, pairs, s);
    case GK_DW: return launch_kind<GK_DW>(ta, tb, to0, to1, p, sms, pairs, s);
  }
  return cudaErrorInvalidValue;
}

}  // namespace moe
