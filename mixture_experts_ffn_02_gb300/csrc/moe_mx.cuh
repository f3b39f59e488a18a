// Device helpers of the MXFP8 path (sm_103a): the e4m3 / UE8M0 block
// quantiser, 32-byte stores, the layout of scale factors in memory, and
// inline-PTX wrappers for the block-scaled tcgen05 MMA and tcgen05.cp on CTA
// pairs.
//
// "KohakUwULLM" README, Key features: MXFP8 = e4m3 values with UE8M0 scales,
// one scale per 32 consecutive values, on the feed-forward pair and the
// routed experts.
#pragma once

#include <cuda_fp8.h>

#include "moe_common.cuh"

namespace moe {

// ----------------------------------------------------------------- quantiser
// One block of 32 values: shared exponent X = floor(log2 max|v|) - 8 (8 is the
// exponent of 448, the largest e4m3 normal), clamped below at -127 (zero and
// fp32-subnormal maxima); the scale byte is X + 127.  Each v * 2^-X (exact: a
// power-of-two scaling of a finite fp32 whose result stays below 512) is
// converted to e4m3 by the hardware conversion, round to nearest even,
// saturating at +-448.  codes[w] holds elements 4w .. 4w+3, lowest first.
__device__ __forceinline__ int mx_block_exp(float amax) {
  const int X = (int)((__float_as_uint(amax) >> 23) & 0xFFu) - 127 - 8;
  return X < -127 ? -127 : X;
}
// Four values times inv (2^-X) as four e4m3 codes, the first lowest.
__device__ __forceinline__ uint32_t mx_cvt4(const float* v, float inv) {
  const uint32_t lo = __nv_cvt_float2_to_fp8x2(make_float2(v[0] * inv, v[1] * inv),
                                               __NV_SATFINITE, __NV_E4M3);
  const uint32_t hi = __nv_cvt_float2_to_fp8x2(make_float2(v[2] * inv, v[3] * inv),
                                               __NV_SATFINITE, __NV_E4M3);
  return (lo & 0xFFFFu) | (hi << 16);
}
__device__ __forceinline__ uint32_t mx_quant32(const float* v, uint32_t* codes) {
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(v[i]));
  const int X = mx_block_exp(amax);
  const float inv = __uint_as_float((uint32_t)(127 - X) << 23);     // 2^-X
#pragma unroll
  for (int w = 0; w < 8; ++w) codes[w] = mx_cvt4(v + 4 * w, inv);
  return (uint32_t)(X + 127);
}
// The same block quantiser when a block of 32 is held 8 values per lane by
// four consecutive lanes (4q .. 4q+3, in element order): the block maximum
// by shuffles among the four, this lane's eight codes in codes[0..1], the
// scale byte returned to all four.  Every lane of the warp must call it.
__device__ __forceinline__ uint32_t mx_quant8x4(const float* v, uint32_t* codes) {
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(v[i]));
  amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
  amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
  const int X = mx_block_exp(amax);
  const float inv = __uint_as_float((uint32_t)(127 - X) << 23);
  codes[0] = mx_cvt4(v, inv);
  codes[1] = mx_cvt4(v + 4, inv);
  return (uint32_t)(X + 127);
}

// 32-byte global store (one full sector per lane); the address must be
// 32-byte aligned.
__device__ __forceinline__ void st_v8(void* p, const uint32_t* v) {
  asm volatile("st.global.v8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};"
               :: "l"(p), "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]),
                  "r"(v[6]), "r"(v[7]) : "memory");
}

// 32 lanes x 64 (128) consecutive 32-bit TMEM columns in one instruction:
// thread i of the warp receives lane (base lane + i), columns [col, col+64).
__device__ __forceinline__ void tmem_ld64(uint32_t taddr, uint32_t* r) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x64.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63}, [%64];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]), "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]), "=r"(r[40]), "=r"(r[41]), "=r"(r[42]), "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]), "=r"(r[48]), "=r"(r[49]), "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55]), "=r"(r[56]), "=r"(r[57]), "=r"(r[58]), "=r"(r[59]), "=r"(r[60]), "=r"(r[61]), "=r"(r[62]), "=r"(r[63])
               : "r"(taddr));
}
__device__ __forceinline__ void tmem_ld128(uint32_t taddr, uint32_t* r) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x128.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63,%64,%65,%66,%67,%68,%69,%70,%71,%72,%73,%74,%75,%76,%77,%78,%79,%80,%81,%82,%83,%84,%85,%86,%87,%88,%89,%90,%91,%92,%93,%94,%95,%96,%97,%98,%99,%100,%101,%102,%103,%104,%105,%106,%107,%108,%109,%110,%111,%112,%113,%114,%115,%116,%117,%118,%119,%120,%121,%122,%123,%124,%125,%126,%127}, [%128];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]), "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]), "=r"(r[40]), "=r"(r[41]), "=r"(r[42]), "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]), "=r"(r[48]), "=r"(r[49]), "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55]), "=r"(r[56]), "=r"(r[57]), "=r"(r[58]), "=r"(r[59]), "=r"(r[60]), "=r"(r[61]), "=r"(r[62]), "=r"(r[63]), "=r"(r[64]), "=r"(r[65]), "=r"(r[66]), "=r"(r[67]), "=r"(r[68]), "=r"(r[69]), "=r"(r[70]), "=r"(r[71]), "=r"(r[72]), "=r"(r[73]), "=r"(r[74]), "=r"(r[75]), "=r"(r[76]), "=r"(r[77]), "=r"(r[78]), "=r"(r[79]), "=r"(r[80]), "=r"(r[81]), "=r"(r[82]), "=r"(r[83]), "=r"(r[84]), "=r"(r[85]), "=r"(r[86]), "=r"(r[87]), "=r"(r[88]), "=r"(r[89]), "=r"(r[90]), "=r"(r[91]), "=r"(r[92]), "=r"(r[93]), "=r"(r[94]), "=r"(r[95]), "=r"(r[96]), "=r"(r[97]), "=r"(r[98]), "=r"(r[99]), "=r"(r[100]), "=r"(r[101]), "=r"(r[102]), "=r"(r[103]), "=r"(r[104]), "=r"(r[105]), "=r"(r[106]), "=r"(r[107]), "=r"(r[108]), "=r"(r[109]), "=r"(r[110]), "=r"(r[111]), "=r"(r[112]), "=r"(r[113]), "=r"(r[114]), "=r"(r[115]), "=r"(r[116]), "=r"(r[117]), "=r"(r[118]), "=r"(r[119]), "=r"(r[120]), "=r"(r[121]), "=r"(r[122]), "=r"(r[123]), "=r"(r[124]), "=r"(r[125]), "=r"(r[126]), "=r"(r[127])
               : "r"(taddr));
}

// ----------------------------------------------------------------- scale layout
// Scale factors sit in 512-byte atoms, one per (128-row block, 128-column
// group): 128 rows x 4 blocks of 32 along K.  Row r, block kb of the atom is
// byte (r % 32) * 16 + (r / 32) * 4 + kb.  tcgen05.cp .32x128b.warpx4 copies
// an atom into 4 TMEM columns, atom row r % 32 to lane r % 32 of all four lane
// quadrants, and the block-scaled MMA reads row (or column) m's scale of the
// K-block given by the instruction's scale-factor id from column base + m / 32,
// byte id, in the lane of m's quadrant.
__host__ __device__ __forceinline__ int mx_sf_byte(int r, int kb) {
  return (r & 31) * 16 + ((r >> 5) & 3) * 4 + kb;
}
constexpr int kMxAtom = 512;

// ----------------------------------------------------------------- tcgen05
// Instruction descriptor of kind::mxf8f6f4 with e4m3 A and B (format 0), fp32
// accumulate, UE8M0 scales (bit 23), both operands K-major; the A and B
// scale-factor ids (the byte of the scale column) at bits 29-30 and 4-5.
__host__ __device__ constexpr uint32_t umma_idesc_mx(int M, int N) {
  return ((uint32_t)(N >> 3) << 17) | (1u << 23) | ((uint32_t)(M >> 4) << 24);
}
__host__ __device__ constexpr uint32_t umma_idesc_sfid(uint32_t idesc, uint32_t id) {
  return idesc | (id << 29) | (id << 4);
}

// CTA-pair form: issued by one thread of the even CTA; A rows 0-127 and D
// lanes in the even CTA, rows 128-255 in the odd one, B columns split in
// halves; each CTA reads its rows' A scales and the scales of all N columns
// of B from its own TMEM at the given addresses.
__device__ __forceinline__ void umma_mx_pair(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc,
                                             uint32_t idesc, uint32_t tsfa, uint32_t tsfb,
                                             uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %6, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::mxf8f6f4.block_scale.scale_vec::1X"
      " [%0], %1, %2, %3, [%4], [%5], p;\n\t}"
      :: "r"(tmem_d), "l"(adesc), "l"(bdesc), "r"(idesc), "r"(tsfa), "r"(tsfb),
         "r"(accumulate)
      : "memory");
}

// Shared-memory descriptor without swizzle (byte offsets >> 4).
__device__ __forceinline__ uint64_t umma_desc_plain(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
  d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
  d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
  d |= (uint64_t)1 << 46;
  return d;
}

// One 512-byte scale atom (32 rows of 16 bytes, contiguous in shared memory)
// into 4 TMEM columns of all 128 lanes; issued by the even CTA of a pair, it
// copies each CTA's atom (same shared offset) into its own TMEM (same
// address), ordered before the MMAs the same thread issues after it.
__device__ __forceinline__ void tmem_cp_atom_pair(uint32_t taddr, uint32_t saddr) {
  asm volatile("tcgen05.cp.cta_group::2.32x128b.warpx4 [%0], %1;"
               :: "r"(taddr), "l"(umma_desc_plain(saddr, 128, 128)) : "memory");
}

}  // namespace moe
