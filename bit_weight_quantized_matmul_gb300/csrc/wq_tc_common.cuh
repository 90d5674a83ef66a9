// wq_tc_common.cuh -- device pieces shared by the tensor-core kernels: per-format
// weight decoding into bf16 pairs for the MMA A operand held in tensor memory.
#pragma once
#include "wq_device.cuh"
#include "wq_internal.h"

namespace wq {
namespace tc {

constexpr int kKS = 64;    // K per pipeline chunk (one 128-byte swizzle row of bf16 x)
constexpr int kRows = 128; // weight rows per tile (the MMA M)

template <int FMT>
struct Fmt {
  static constexpr bool BYTE = FMT == WQ_Q8_0 || FMT == WQ_FP8;   // one byte per weight
  static constexpr bool UNIT = FMT == WQ_Q5_0 || FMT == WQ_Q4_1;  // 80-byte units of 128 weights
  static constexpr int WB = BYTE ? 64 : UNIT ? 40 : 32;             // packed bytes per row per 64 weights
  // bytes per row and 64-block of the per-block scales staged for a tile (FP8: none, its one
  // scale per row is applied in the epilogue; q4_1: none, its scales travel in the units)
  static constexpr int SCB = FMT == WQ_NF4 ? 1 : (FMT == WQ_FP8 || FMT == WQ_Q4_1) ? 0 : 4;
};

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&v)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]), "r"(v[9]),
      "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15]), "r"(v[16]), "r"(v[17]), "r"(v[18]),
      "r"(v[19]), "r"(v[20]), "r"(v[21]), "r"(v[22]), "r"(v[23]), "r"(v[24]), "r"(v[25]), "r"(v[26]), "r"(v[27]),
      "r"(v[28]), "r"(v[29]), "r"(v[30]), "r"(v[31])
      : "memory");
}

// Byte -> (value of low nibble, value of high nibble) for the 4-bit formats.
template <int FMT>
__device__ __forceinline__ float nibble_value(uint32_t c) {
  if (FMT == WQ_NF4) return kNF4[c];
  if (FMT == WQ_Q4_0) return (float)((int)c - 8);
  if (FMT == WQ_Q4_1) return (float)c;
  if (FMT == WQ_Q5_0) return (float)((int)c - 16);  // the fifth bit adds 16 afterwards
  return kE2M1[c];  // NVFP4: E2M1 value; the E4M3 block scale multiplies it, g is applied on D
}

__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&v)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]), "r"(v[9]),
      "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15])
      : "memory");
}

// The per-(row, 64-chunk) scale word staged in shared memory for the dequant warps:
//   NF4         the decoded block absmax a_hat = q * s2 + offset (fp32 bits; one 64-block per chunk)
//   NVFP4       the four E4M3 block-scale bytes of the chunk (one per 16 elements)
//   q4_0, q8_0  the two fp16 d of the chunk (one per 32 elements)
// For the last three the word is the 4 bytes at offset n*K/16 + 4c of the scales blob.
template <int FMT>
__device__ __forceinline__ uint32_t scale_word(const uint8_t* __restrict__ scales, const ScalesLayout& lay,
                                               int64_t K, int64_t n, int64_t c) {
  if (FMT == WQ_NF4) {
    const int64_t b = n * (K / 64) + c;
    const int8_t q = reinterpret_cast<const int8_t*>(scales)[b];
    const float s2 = reinterpret_cast<const float*>(scales + lay.s2_off)[b / 256];
    const float off = *reinterpret_cast<const float*>(scales + lay.offset_off);
    return __float_as_uint(__fadd_rn(__fmul_rn((float)q, s2), off));
  }
  return *reinterpret_cast<const uint32_t*>(scales + n * (K / 16) + 4 * c);
}

// Decode NE (32 or 64) consecutive weights of one 64-element block of a row into NE/2
// bf16x2 words.  `part` selects which NE-element part of the block (0 when NE == 64);
// `sword` is the block's scale word (see scale_word); `wv` holds the NE packed codes
// (16 bytes per entry, already loaded from shared memory).  The byte -> (value, value) table holds LUTREP copies
// interleaved so that lane group `lsel` reads its own banks (LUTREP = 16: the 16
// lanes of a half-warp never collide on a 64-bit load, whatever the codes).
template <int FMT, int NE, int LUTREP>
__device__ __forceinline__ void decode_span(uint32_t sword, int part, const uint4* wv, const float2* lut,
                                            int lsel, uint32_t (&out)[NE / 2]) {
  static_assert(NE == 32 || NE == 64, "span");
  if (FMT == WQ_Q8_0) {
#pragma unroll
    for (int q = 0; q < NE / 16; ++q) {
      const int e0 = part * NE + q * 16;  // element index within the 64-block
      const float d = f16_bits_to_f32(e0 < 32 ? (sword & 0xFFFFu) : (sword >> 16));
      const uint4 v = wv[q];
      const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float a0 = (float)(int8_t)(u[j] & 0xFF), a1 = (float)(int8_t)((u[j] >> 8) & 0xFF);
        const float a2 = (float)(int8_t)((u[j] >> 16) & 0xFF), a3 = (float)(int8_t)(u[j] >> 24);
        out[q * 8 + j * 2] = pack_bf16x2(__fmul_rn(a0, d), __fmul_rn(a1, d));
        out[q * 8 + j * 2 + 1] = pack_bf16x2(__fmul_rn(a2, d), __fmul_rn(a3, d));
      }
    }
    return;
  }
#pragma unroll
  for (int q = 0; q < NE / 32; ++q) {
    const uint4 v = wv[q];
    const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int e0 = part * NE + q * 32 + j * 8;  // first element of this word within the 64-block
      float s;
      if (FMT == WQ_NF4) s = __uint_as_float(sword);
      else if (FMT == WQ_Q4_0) s = f16_bits_to_f32(e0 < 32 ? (sword & 0xFFFFu) : (sword >> 16));
      else s = e4m3_to_f32((sword >> (8 * (e0 / 16))) & 0xFFu);
#pragma unroll
      for (int b = 0; b < 4; ++b) {
        const float2 lv = lut[((u[j] >> (8 * b)) & 0xFFu) * LUTREP + lsel];
        out[q * 16 + j * 4 + b] = pack_bf16x2(__fmul_rn(lv.x, s), __fmul_rn(lv.y, s));
      }
    }
  }
}

__device__ __forceinline__ void tmem_st_n(uint32_t taddr, const uint32_t (&v)[16]) { tmem_st16(taddr, v); }
__device__ __forceinline__ void tmem_st_n(uint32_t taddr, const uint32_t (&v)[32]) { tmem_st32(taddr, v); }

// Byte -> packed bf16 pair (value of the low nibble in the low half).  NF4 values are
// rounded to bf16 here; q4_0's (q - 8) and NVFP4's E2M1 values are exact in bf16.
template <int FMT>
__device__ __forceinline__ uint32_t nibble_pair_bf16(uint32_t byte) {
  return pack_bf16x2(nibble_value<FMT>(byte & 15u), nibble_value<FMT>(byte >> 4));
}

__device__ __forceinline__ uint32_t hmul2_bf16(uint32_t a, uint32_t b) {
  __nv_bfloat162 x = *reinterpret_cast<__nv_bfloat162*>(&a);
  __nv_bfloat162 y = *reinterpret_cast<__nv_bfloat162*>(&b);
  __nv_bfloat162 r = __hmul2(x, y);
  return *reinterpret_cast<uint32_t*>(&r);
}

// Decode NE elements of one 64-element block with a bf16-pair table (LUTREP copies,
// `lsel` = this lane's copy).  SCALED: multiply each pair by the block's NVFP4 E4M3
// scale in bf16 (exact: an E2M1 value times an E4M3 value has at most 5 significant
// bits).  Unscaled (the per-block scale is applied to the MMA partial sums
// afterwards): NF4 codebook values in bf16, q4_0 (q - 8), q8_0 q -- the last two exact.
template <int FMT, int NE, int LUTREP, bool SCALED>
__device__ __forceinline__ void decode_span_bf16(uint32_t sword, int part, const uint4* wv,
                                                 const uint32_t* lut, int lsel, uint32_t (&out)[NE / 2]) {
  static_assert(NE == 32 || NE == 64, "span");
  if (FMT == WQ_Q8_0) {
#pragma unroll
    for (int q = 0; q < NE / 16; ++q) {
      const uint4 v = wv[q];
      const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        out[q * 8 + j * 2] = pack_bf16x2((float)(int8_t)(u[j] & 0xFF), (float)(int8_t)((u[j] >> 8) & 0xFF));
        out[q * 8 + j * 2 + 1] = pack_bf16x2((float)(int8_t)((u[j] >> 16) & 0xFF), (float)(int8_t)(u[j] >> 24));
      }
    }
    return;
  }
  // this lane's copy of the table, addressed in bytes: one byte-permute and one shifted add
  // per packed byte
  const uint8_t* lbase = reinterpret_cast<const uint8_t*>(lut + lsel);
#pragma unroll
  for (int q = 0; q < NE / 32; ++q) {
    const uint4 v = wv[q];
    const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      uint32_t spair = 0u;
      if (SCALED) {
        const int e0 = part * NE + q * 32 + j * 8;
        const uint32_t sb = __float_as_uint(e4m3_to_f32((sword >> (8 * (e0 / 16))) & 0xFFu)) >> 16;
        spair = sb | (sb << 16);  // E4M3 values are exact in bf16
      }
#pragma unroll
      for (int b = 0; b < 4; ++b) {
        const uint32_t byte = __byte_perm(u[j], 0u, 0x4440u + (uint32_t)b);
        const uint32_t pair = *reinterpret_cast<const uint32_t*>(lbase + byte * (uint32_t)(LUTREP * 4));
        out[q * 16 + j * 4 + b] = SCALED ? hmul2_bf16(pair, spair) : pair;
      }
    }
  }
}

}  // namespace tc
}  // namespace wq

namespace wq {
namespace tc {
// 16-byte chunk `ck` of weight row `r` in a pipeline stage made of NBOX TMA boxes
// [128 rows x RB bytes], each written with the TMA swizzle of width RB (32/64/128 B:
// address bits [4, 4+log2(RB/16)) XOR bits [7, ...)), which keeps the 32 rows a warp
// reads on distinct banks.
template <int RB, int NBOX>
__device__ __forceinline__ uint4 load_wchunk(const uint8_t* stage, int r, int ck) {
  constexpr int CPB = RB / 16;  // chunks per box row
  constexpr uint32_t mask = RB == 128 ? 7u : RB == 64 ? 3u : 1u;
  const int box = (NBOX > 1) ? ck / CPB : 0;
  uint32_t off = (uint32_t)(r * RB + (ck % CPB) * 16);
  off ^= ((off >> 7) & mask) << 4;
  return *reinterpret_cast<const uint4*>(stage + box * (128 * RB) + off);
}

template <int RB>
constexpr CUtensorMapSwizzle swizzle_of() {
  return RB == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : RB == 64 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_32B;
}
}  // namespace tc
}  // namespace wq

namespace wq {
namespace tc {
__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
  return d;
}

// Eight E2M1 codes (nibbles of u, element 2j in the low nibble of byte j) -> four packed bf16
// pairs, without tables in memory.  The 3-bit magnitude of a code indexes the 8 bytes of two
// registers in one byte permute: the high and the low bytes of the bf16 values of
// {0, .5, 1, 1.5, 2, 3, 4, 6} are 00 3F 3F 3F 40 40 40 40 and 00 00 80 C0 00 40 80 C0.  The sign
// bits of four codes at a time go into the msbs of their high bytes before the bytes are paired: a
// sign-replicating selector picks, for high byte k, the byte of u or of u << 4 whose msb is code k's
// sign (u << 4 moves each low nibble's sign bit to its byte's msb).  X2P120: every value times 2^120
// (high bytes 00 7B 7B 7B 7C 7C 7C 7C), the partner of e4m3_bf16pair_m120.
template <bool X2P120 = false>
__device__ __forceinline__ void e2m1x8_to_bf16(uint32_t u, uint32_t (&w)[4]) {
  constexpr uint32_t H0 = X2P120 ? 0x7B7B7B00u : 0x3F3F3F00u, H1 = X2P120 ? 0x7C7C7C7Cu : 0x40404040u;
  constexpr uint32_t L0 = 0xC0800000u, L1 = 0xC0804000u;
  const uint32_t sa = u & 0x7777u, sb = (u >> 16) & 0x7777u;
  const uint32_t u4 = u << 4;
  const uint32_t hiA = prmt(H0, H1, sa) | (prmt(u, u4, 0x9D8Cu) & 0x80808080u);  // codes 0..3
  const uint32_t hiB = prmt(H0, H1, sb) | (prmt(u, u4, 0xBFAEu) & 0x80808080u);  // codes 4..7
  const uint32_t loA = prmt(L0, L1, sa), loB = prmt(L0, L1, sb);
  w[0] = prmt(loA, hiA, 0x5140u);
  w[1] = prmt(loA, hiA, 0x7362u);
  w[2] = prmt(loB, hiB, 0x5140u);
  w[3] = prmt(loB, hiB, 0x7362u);
}

// x: an E4M3 code in bits 0..7 and again in bits 16..23 (zeros elsewhere).  Returns, in both bf16
// halves, the code's value times 2^-120: its sign, exponent and mantissa fields moved to bf16's places
// (exponent field e, mantissa m << 4).  Exact for every code, the subnormal codes landing on bf16
// subnormals with the same mantissa; times an E2M1 value scaled by 2^120 the bf16 product is the
// exact e2m1 * e4m3 (at most 5 significant bits, within bf16's normal range).
__device__ __forceinline__ uint32_t e4m3_bf16pair_m120(uint32_t x) {
  return ((x << 4) & 0x07F007F0u) | ((x << 8) & 0x80008000u);
}

// NVFP4: decode NE elements of one 64-element block with E2M1 -> bf16 in registers and the
// block's E4M3 scales applied as an exact bf16 product.
template <int NE>
__device__ __forceinline__ void decode_span_nvfp4_reg(uint32_t sword, int part, const uint4* wv,
                                                      uint32_t (&out)[NE / 2]) {
#pragma unroll
  for (int q = 0; q < NE / 32; ++q) {
    const uint32_t u[4] = {wv[q].x, wv[q].y, wv[q].z, wv[q].w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int e0 = part * NE + q * 32 + j * 8;
      const uint32_t spair = e4m3_bf16pair_m120(prmt(sword, 0u, 0x4040u + 0x0101u * (e0 / 16)));
      uint32_t w[4];
      e2m1x8_to_bf16<true>(u[j], w);
#pragma unroll
      for (int b = 0; b < 4; ++b) out[q * 16 + j * 4 + b] = hmul2_bf16(w[b], spair);
    }
  }
}
}  // namespace tc
}  // namespace wq

namespace wq {
namespace tc {
__device__ __forceinline__ void epi_bar() { asm volatile("bar.sync 1, 128;" ::: "memory"); }

// Store one 16-column slab of a D tile (TMEM lanes = 128 weight rows n0.., columns = 16
// activation rows m0..) to y[M, N] bf16 through shared memory: each of the 128 epilogue
// threads (its TMEM lane r) scales and writes its 16 values into stage[m][r], then the
// threads copy the [16 x 128] bf16 slab out as whole 256-byte rows with 16-byte stores.
// `stage` is this slab's 4 KB buffer; callers alternate two buffers (one barrier per slab).
__device__ __forceinline__ void store_slab_bf16(const float (&acc)[16], float gsc, float bval, int r,
                                                uint16_t* stage, void* y, int64_t M, int64_t N, int64_t m0,
                                                int64_t n0) {
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    const float v = __fadd_rn(__fmul_rn(acc[j], gsc), bval);
    stage[j * 128 + r] = __bfloat16_as_ushort(__float2bfloat16_rn(v));
  }
  epi_bar();
  // thread t copies 16 elements: row t / 8, columns (t % 8) * 16 .. + 15
  const int row = r >> 3, seg = (r & 7) * 16;
  const int64_t m = m0 + row, n = n0 + seg;
  if (m < M && n < N) {
    __nv_bfloat16* dst = reinterpret_cast<__nv_bfloat16*>(y) + m * N + n;
    const uint16_t* src = stage + row * 128 + seg;
    if (n + 16 <= N && (N & 7) == 0) {
      const uint4* s4 = reinterpret_cast<const uint4*>(src);
      uint4* d4 = reinterpret_cast<uint4*>(dst);
      d4[0] = s4[0];
      d4[1] = s4[1];
    } else {
      for (int e = 0; e < 16 && n + e < N; ++e) reinterpret_cast<uint16_t*>(dst)[e] = src[e];
    }
  }
}
}  // namespace tc
}  // namespace wq

namespace wq {
namespace tc {
// FP8 E4M3: decode NE codes (one byte each) into exact bf16 pairs.  The E4M3 sign, exponent and
// mantissa fields placed at the bf16 bit positions (exponent field unchanged, mantissa shifted up
// by four) make the bf16 number E4M3(code) * 2^-120, subnormals included (an E4M3 subnormal lands
// on a bf16 subnormal with the same significand), and one bf16 multiply by 2^120 restores the
// value exactly.  The per-row scale is applied to the fp32 accumulator in the epilogue.
__device__ __forceinline__ uint32_t e4m3x2_to_bf16x2(uint32_t spread) {  // bytes in bits [0,8), [16,24)
  const uint32_t bits = ((spread << 4) & 0x07F007F0u) | ((spread << 8) & 0x80008000u);
  return hmul2_bf16(bits, 0x7B807B80u);  // x 2^120 in both halves
}

template <int NE>
__device__ __forceinline__ void decode_span_fp8(const uint4* wv, uint32_t (&out)[NE / 2]) {
#pragma unroll
  for (int q = 0; q < NE / 16; ++q) {
    const uint32_t u[4] = {wv[q].x, wv[q].y, wv[q].z, wv[q].w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      out[q * 8 + j * 2] = e4m3x2_to_bf16x2(prmt(u[j], 0u, 0x4140u));
      out[q * 8 + j * 2 + 1] = e4m3x2_to_bf16x2(prmt(u[j], 0u, 0x4342u));
    }
  }
}
}  // namespace tc
}  // namespace wq

namespace wq {
namespace tc {
// q4_1 / q5_0: decode elements [64h, 64h + 64) of a 128-element unit into 32 bf16 pairs: `nib` the
// 32 bytes of their nibbles, `side` the unit's 8 side-data bytes of its blocks 2h and 2h + 1 (q5_0:
// fifth bits, bit e = element e of the block; q4_1: the blocks' (fp16 d, fp16 m)), `sword` (q5_0)
// the two blocks' fp16 d.  The fp32 value is the one wq_dequant gives (q5_0 (q - 16) * d; q4_1
// q * d + m), rounded once to bf16 for the MMA.
template <int FMT, int LUTREP>
__device__ __forceinline__ void decode_unit64(const uint4 (&nib)[2], uint2 side, uint32_t sword, const float2* lut,
                                              int lsel, uint32_t (&out)[32]) {
#pragma unroll
  for (int blk = 0; blk < 2; ++blk) {
    const uint32_t sd = blk ? side.y : side.x;
    float d, madd = 0.0f;
    if (FMT == WQ_Q4_1) {
      d = f16_bits_to_f32(sd & 0xFFFFu);
      madd = f16_bits_to_f32(sd >> 16);
    } else {
      d = f16_bits_to_f32(blk ? (sword >> 16) : (sword & 0xFFFFu));
    }
    const uint4 v = nib[blk];
    const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
#pragma unroll
      for (int b = 0; b < 4; ++b) {
        const int e = j * 8 + b * 2;  // element within the block
        const float2 lv = lut[((u[j] >> (8 * b)) & 0xFFu) * LUTREP + lsel];
        float v0, v1;
        if (FMT == WQ_Q5_0) {
          v0 = __fmul_rn(__fadd_rn(lv.x, ((sd >> e) & 1u) ? 16.0f : 0.0f), d);
          v1 = __fmul_rn(__fadd_rn(lv.y, ((sd >> (e + 1)) & 1u) ? 16.0f : 0.0f), d);
        } else {
          v0 = __fadd_rn(__fmul_rn(lv.x, d), madd);
          v1 = __fadd_rn(__fmul_rn(lv.y, d), madd);
        }
        out[blk * 16 + j * 4 + b] = pack_bf16x2(v0, v1);
      }
    }
  }
}
}  // namespace tc
}  // namespace wq
