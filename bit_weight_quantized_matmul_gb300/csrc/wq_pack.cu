// wq_pack.cu -- GPU packers, the decode-to-fp32 export and the NVFP4 runtime
// activation quantiser.  Every quantiser step is one IEEE fp32 operation
// (__fdiv_rn / __fmul_rn / __fadd_rn / __fsub_rn, rintf = round half to even),
// so the bytes are identical to a plain sequential evaluation of the block
// definitions.
//
// Sources: PR "asr: add a 4-bit nf4 option for the Whisper engine", "What's
// here" (NF4 + double-quant); model card "whisper-large-v3-turbo -- NVFP4",
// "What is quantized" (E2M1 per 16, E4M3 block scale, fp32 global scale,
// runtime activation quantisation); PR "Run quantized Whisper on the fused
// Metal decode path", "Summary" (q4_0 / q8_0 blocks of 32 with an fp16 d).
#include <cuda_runtime.h>

#include <mutex>

#include "wq_device.cuh"
#include "wq_internal.h"

namespace wq {
namespace {

constexpr int kNF4Block = 64;
constexpr int kDQGroup = 256;
constexpr int kNVBlock = 16;
constexpr int kGGBlock = 32;

inline int grid_for(int64_t n, int threads) {
  int64_t g = (n + threads - 1) / threads;
  return (int)(g < 1 ? 1 : g);
}

// ------------------------------------------------------------------ NF4
// 1) per 64-block absmax -> fp32, parked in the (not yet written) packed buffer.
__global__ void nf4_absmax_kernel(const float* __restrict__ W, int64_t nb, float* __restrict__ tmp) {
  const int64_t b = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (b >= nb) return;
  const float4* src = reinterpret_cast<const float4*>(W + b * kNF4Block);
  float a = 0.0f;
#pragma unroll
  for (int i = 0; i < kNF4Block / 4; ++i) {
    const float4 v = src[i];
    a = fmaxf(a, fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w))));
  }
  tmp[b] = a;
}

// Exact sum of non-negative fp32 values kept as per-exponent integer mantissa
// sums, converted once to fp64 with round-to-nearest-even.
// total = sum_e bucket[e] * 2^(e - 150), e = biased exponent (subnormals use e = 1).
__device__ double exact_bucket_sum_to_double(const unsigned long long* bucket) {
  unsigned long long L[7] = {0, 0, 0, 0, 0, 0, 0};  // B = total * 2^149, 448 bits
  for (int e = 1; e < 255; ++e) {
    const unsigned long long v = bucket[e];
    if (!v) continue;
    const int sh = e - 1, li = sh >> 6, bi = sh & 63;
    const unsigned long long lo = v << bi;
    const unsigned long long hi = bi ? (v >> (64 - bi)) : 0ull;
    unsigned long long old = L[li];
    L[li] += lo;
    unsigned long long add = hi + (L[li] < old ? 1ull : 0ull);
    for (int j = li + 1; add && j < 7; ++j) {
      old = L[j];
      L[j] += add;
      add = (L[j] < old) ? 1ull : 0ull;
    }
  }
  int top = -1;
  for (int i = 6; i >= 0; --i)
    if (L[i]) { top = i * 64 + 63 - __clzll((long long)L[i]); break; }
  if (top < 0) return 0.0;
  if (top <= 52) return ldexp((double)L[0], -149);
  int sh = top - 52;  // keep bits [sh, top]
  const int li = sh >> 6, bi = sh & 63;
  unsigned long long mant = L[li] >> bi;
  if (bi && li + 1 < 7) mant |= L[li + 1] << (64 - bi);
  mant &= (1ull << 53) - 1;
  const int rp = sh - 1;  // rounding bit position
  const unsigned long long rnd = (L[rp >> 6] >> (rp & 63)) & 1ull;
  bool sticky = (L[rp >> 6] & ((1ull << (rp & 63)) - 1ull)) != 0ull;
  for (int i = 0; i < (rp >> 6); ++i) sticky = sticky || (L[i] != 0ull);
  if (rnd && (sticky || (mant & 1ull))) {
    ++mant;
    if (mant >> 53) { mant >>= 1; ++sh; }
  }
  return ldexp((double)mant, sh - 149);
}

// Adds absmax value i (none when i >= nb) to the per-exponent mantissa sums; all 32 lanes of the
// warp call it together.
__device__ __forceinline__ void bucket_add(const float* tmp, int64_t nb, int64_t i, unsigned long long* bucket) {
  uint32_t e = 1, m = 0;
  if (i < nb) {
    const uint32_t bits = __float_as_uint(tmp[i]);
    e = bits >> 23;
    m = bits & 0x7FFFFFu;
    if (e) m |= 0x800000u; else e = 1;
  }
  const unsigned mask = __match_any_sync(0xFFFFFFFFu, e);
  const unsigned sum = __reduce_add_sync(mask, m);  // <= 32 * 2^24 fits 32 bits
  if ((int)(threadIdx.x & 31) == __ffs(mask) - 1 && sum) atomicAdd(&bucket[e], (unsigned long long)sum);
}

// Group g of 256 absmax values, one warp: t = a - offset, s2 = max|t| / 127,
// q = clamp(rint(t / s2), -127, 127).
__device__ __forceinline__ void dq_group(const float* tmp, int64_t nb, float off, int64_t g, int lane,
                                         int8_t* absmax_q, float* s2_out) {
  float t[kDQGroup / 32];
  uint32_t mx = 0;
#pragma unroll
  for (int j = 0; j < kDQGroup / 32; ++j) {
    const int64_t i = g * kDQGroup + j * 32 + lane;
    t[j] = (i < nb) ? __fsub_rn(tmp[i], off) : 0.0f;
    const uint32_t ab = __float_as_uint(fabsf(t[j]));
    mx = (i < nb && ab > mx) ? ab : mx;
  }
  mx = __reduce_max_sync(0xFFFFFFFFu, mx);
  const float s2 = __fdiv_rn(__uint_as_float(mx), 127.0f);
  if (lane == 0) s2_out[g] = s2;
#pragma unroll
  for (int j = 0; j < kDQGroup / 32; ++j) {
    const int64_t i = g * kDQGroup + j * 32 + lane;
    if (i < nb) {
      float q = 0.0f;
      if (s2 != 0.0f) q = fminf(fmaxf(rintf(__fdiv_rn(t[j], s2)), -127.0f), 127.0f);
      absmax_q[i] = (int8_t)(int)q;
    }
  }
}

// 2) one CTA: offset = fp32(exact_sum(absmax) / count); per group of 256:
//    t = a - offset, s2 = max|t| / 127, q = clamp(rint(t / s2), -127, 127).
__global__ void __launch_bounds__(1024) nf4_double_quant_kernel(const float* __restrict__ tmp, int64_t nb,
                                                                int8_t* __restrict__ absmax_q,
                                                                float* __restrict__ s2_out,
                                                                float* __restrict__ offset_out,
                                                                int64_t pad_end) {
  __shared__ unsigned long long bucket[256];
  __shared__ float s_offset;
  const int tid = threadIdx.x;
  for (int i = tid; i < 256; i += blockDim.x) bucket[i] = 0ull;
  __syncthreads();
  for (int64_t base = 0; base < nb; base += blockDim.x) bucket_add(tmp, nb, base + tid, bucket);
  __syncthreads();
  if (tid == 0) {
    const double total = exact_bucket_sum_to_double(bucket);
    const float off = __double2float_rn(__ddiv_rn(total, (double)nb));
    s_offset = off;
    *offset_out = off;
    for (int64_t p = nb; p < pad_end; ++p) absmax_q[p] = 0;
  }
  __syncthreads();
  const float off = s_offset;
  const int warp = tid >> 5, lane = tid & 31, nwarps = blockDim.x >> 5;
  const int64_t ng = (nb + kDQGroup - 1) / kDQGroup;
  for (int64_t g = warp; g < ng; g += nwarps) dq_group(tmp, nb, off, g, lane, absmax_q, s2_out);
}

// 2') the same in parallel: per-CTA bucket sums added into global buckets, one thread for the offset,
// then one warp per group of 256.
__global__ void __launch_bounds__(1024) nf4_bucket_kernel(const float* __restrict__ tmp, int64_t nb,
                                                          unsigned long long* __restrict__ gbucket) {
  __shared__ unsigned long long bucket[256];
  const int tid = threadIdx.x;
  for (int i = tid; i < 256; i += blockDim.x) bucket[i] = 0ull;
  __syncthreads();
  for (int64_t base = (int64_t)blockIdx.x * blockDim.x; base < nb; base += (int64_t)gridDim.x * blockDim.x)
    bucket_add(tmp, nb, base + tid, bucket);
  __syncthreads();
  for (int i = tid; i < 256; i += blockDim.x)
    if (bucket[i]) atomicAdd(&gbucket[i], bucket[i]);
}

__global__ void nf4_offset_kernel(const unsigned long long* __restrict__ gbucket, int64_t nb,
                                  float* __restrict__ offset_out, int8_t* __restrict__ absmax_q, int64_t pad_end) {
  if (threadIdx.x == 0) *offset_out = __double2float_rn(__ddiv_rn(exact_bucket_sum_to_double(gbucket), (double)nb));
  for (int64_t p = nb + threadIdx.x; p < pad_end; p += blockDim.x) absmax_q[p] = 0;
}

__global__ void nf4_dq_groups_kernel(const float* __restrict__ tmp, int64_t nb, const float* __restrict__ offset,
                                     int8_t* __restrict__ absmax_q, float* __restrict__ s2_out) {
  const int64_t g = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  if (g >= (nb + kDQGroup - 1) / kDQGroup) return;
  dq_group(tmp, nb, *offset, g, threadIdx.x & 31, absmax_q, s2_out);
}

// 3) codes: v = w / absmax (0 for an all-zero block); code = #{midpoints < v}.
__global__ void nf4_codes_kernel(const float* __restrict__ W, int64_t nb, uint8_t* __restrict__ packed) {
  __shared__ float mids[15];
  if (threadIdx.x < 15)
    mids[threadIdx.x] = __fmul_rn(__fadd_rn(kNF4[threadIdx.x], kNF4[threadIdx.x + 1]), 0.5f);
  __syncthreads();
  const int64_t b = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (b >= nb) return;
  const float4* src = reinterpret_cast<const float4*>(W + b * kNF4Block);
  float a = 0.0f;
#pragma unroll
  for (int i = 0; i < kNF4Block / 4; ++i) {
    const float4 v = src[i];
    a = fmaxf(a, fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w))));
  }
  uint4* dst = reinterpret_cast<uint4*>(packed + b * (kNF4Block / 2));
#pragma unroll
  for (int q = 0; q < 2; ++q) {  // 32 elements -> 16 bytes per store
    uint32_t word[4];
#pragma unroll
    for (int w = 0; w < 4; ++w) {
      uint32_t acc = 0;
      const float4 v0 = src[q * 8 + w * 2], v1 = src[q * 8 + w * 2 + 1];
      const float vals[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const float v = (a == 0.0f) ? 0.0f : __fdiv_rn(vals[j], a);
        uint32_t code = 0;
#pragma unroll
        for (int k = 0; k < 15; ++k) code += (mids[k] < v) ? 1u : 0u;
        acc |= code << (4 * j);
      }
      word[w] = acc;
    }
    dst[q] = make_uint4(word[0], word[1], word[2], word[3]);
  }
}

// ------------------------------------------------------------------ NVFP4
// Eight consecutive values (index i, i % 8 == 0) as fp32, with 16-byte vector loads.
__device__ __forceinline__ void load8_f32(const float* p, int64_t i, float (&v)[8]) {
  const float4 a = reinterpret_cast<const float4*>(p + i)[0], b = reinterpret_cast<const float4*>(p + i)[1];
  v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w; v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}
__device__ __forceinline__ void load8_f32(const uint16_t* p, int64_t i, float (&v)[8]) {
  const uint4 a = *reinterpret_cast<const uint4*>(p + i);
  const uint32_t u[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    v[2 * j] = bf16_bits_to_f32(u[j] & 0xFFFFu);
    v[2 * j + 1] = bf16_bits_to_f32(u[j] >> 16);
  }
}

// amax over n values (n % 8 == 0) -> atomicMax on the bit pattern (non-negative floats order as integers)
template <typename T>
__global__ void amax_kernel(const T* __restrict__ X, int64_t n, unsigned* __restrict__ slot) {
  griddep_launch_dependents();  // the quantiser may start loading its blocks
  float a = 0.0f;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x * 8;
  int64_t i = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) * 8;
  // four independent 16-byte loads in flight per thread: the grid is capped at two CTAs per SM
  for (; i + 3 * stride < n; i += 4 * stride) {
    float v0[8], v1[8], v2[8], v3[8];
    load8_f32(X, i, v0);
    load8_f32(X, i + stride, v1);
    load8_f32(X, i + 2 * stride, v2);
    load8_f32(X, i + 3 * stride, v3);
#pragma unroll
    for (int j = 0; j < 8; ++j)
      a = fmaxf(a, fmaxf(fmaxf(fabsf(v0[j]), fabsf(v1[j])), fmaxf(fabsf(v2[j]), fabsf(v3[j]))));
  }
  for (; i < n; i += stride) {
    float v[8];
    load8_f32(X, i, v);
#pragma unroll
    for (int j = 0; j < 8; ++j) a = fmaxf(a, fabsf(v[j]));
  }
  // block maximum first, then one atomic per block
  __shared__ unsigned wmax[32];
  unsigned u = __reduce_max_sync(0xFFFFFFFFu, __float_as_uint(a));
  if ((threadIdx.x & 31) == 0) wmax[threadIdx.x >> 5] = u;
  __syncthreads();
  if (threadIdx.x < 32) {
    u = (threadIdx.x < (blockDim.x >> 5)) ? wmax[threadIdx.x] : 0u;
    u = __reduce_max_sync(0xFFFFFFFFu, u);
    if (threadIdx.x == 0 && u) atomicMax(slot, u);
  }
}

__device__ __forceinline__ float nvfp4_g_from_amax(float amax) {
  return amax == 0.0f ? 1.0f : __fdiv_rn(amax, 2688.0f);
}

// x / S rounded to nearest even, for the 16 elements of a block sharing one S > 0: Markstein's
// division (P. Markstein, "Computation of elementary functions on the IBM RISC System/6000
// processor", IBM J. Res. Dev. 34(1), 1990; Handbook of Floating-Point Arithmetic, ch. 5): with
// y = RN(1/S), q = RN(x * y) and the residual r = x - q * S (exact in one FMA), RN(q + r * y) is
// RN(x / S) while no intermediate leaves the normal range.  One correctly rounded reciprocal per
// block and a few operations per element instead of a full division each; blocks whose S lies
// outside [2^-100, 2^100] take the plain division.  Only the E2M1 code of the quotient is used, so
// quotients past 8 (all saturating) are returned as +-8.
__device__ __forceinline__ void div_block(const float (&v)[16], float S, float (&q)[16]) {
  if (S > 7.888609e-31f && S < 1.2676506e30f) {
    const float y = __frcp_rn(S);
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const float q0 = __fmul_rn(v[i], y);
      const float r = __fmaf_rn(-q0, S, v[i]);
      // the quotient keeps x's sign (a -0 or a negative that rounds to zero stays negative); past
      // |8| every E2M1 code saturates, which also covers a product that overflowed
      const float qc = fabsf(q0) > 8.0f ? 8.0f : fabsf(__fmaf_rn(r, y, q0));
      q[i] = copysignf(qc, v[i]);
    }
  } else {
#pragma unroll
    for (int i = 0; i < 16; ++i) q[i] = __fdiv_rn(v[i], S);
  }
}

// one thread per 16-block along a row: s = e4m3((amax_b / 6) / g), S = dec(s) * g,
// code = e2m1(x / S) (0 where S == 0).  g_src holds amax (g_is_amax) or g itself.
template <typename T>
__global__ void nvfp4_quant_kernel(const T* __restrict__ X, int64_t nblk, const float* __restrict__ g_src,
                                   int g_is_amax, uint8_t* __restrict__ codes, uint8_t* __restrict__ sf,
                                   float* __restrict__ g_copy_out) {
  const int64_t b = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  // a consumer launched with programmatic dependent launch (the W4A4 GEMM with static weights) may
  // start its set-up and weight stream now; it waits for this grid before reading the activations
  griddep_launch_dependents();
  // dynamic g: this kernel runs right after the amax kernel (programmatic dependent launch); x does
  // not depend on it, so the block's values are loaded first and the amax read after the wait
  float v[kNVBlock];
  if (b < nblk) {
    float lo[8], hi[8];
    load8_f32(X, b * kNVBlock, lo);
    load8_f32(X, b * kNVBlock + 8, hi);
#pragma unroll
    for (int i = 0; i < 8; ++i) { v[i] = lo[i]; v[i + 8] = hi[i]; }
  }
  if (g_is_amax) griddep_wait();
  const float gs = *g_src;
  const float g = g_is_amax ? nvfp4_g_from_amax(gs) : gs;
  if (b == 0 && g_copy_out) *g_copy_out = g;
  if (b >= nblk) return;
  float amax = 0.0f;
#pragma unroll
  for (int i = 0; i < kNVBlock; ++i) amax = fmaxf(amax, fabsf(v[i]));
  const uint32_t s = f32_to_e4m3_cvt(__fdiv_rn(__fdiv_rn(amax, 6.0f), g));
  const float S = __fmul_rn(e4m3_to_f32(s), g);
  uint32_t lo = 0, hi = 0;
  if (S != 0.0f) {  // a block whose scale underflows to zero keeps codes 0
    float q[kNVBlock];
    div_block(v, S, q);
    lo = f32x8_to_e2m1x8(q);
    hi = f32x8_to_e2m1x8(q + 8);
  }
  reinterpret_cast<uint2*>(codes)[b] = make_uint2(lo, hi);
  sf[b] = (uint8_t)s;
}

// slot: amax -> g; zero the pad bytes between the block scales and g.
__global__ void nvfp4_finalize_kernel(float* slot, uint8_t* pad_begin, int pad_len) {
  griddep_launch_dependents();
  griddep_wait();  // launched right after the quantiser, which still reads the slot as amax
  if (threadIdx.x == 0) *slot = nvfp4_g_from_amax(*slot);
  if ((int)threadIdx.x < pad_len) pad_begin[threadIdx.x] = 0;
}

// ------------------------------------------------------------------ q4_0 / q8_0
// zero the bytes between the last fp16 d and the 16-byte aligned end of the scales blob
__device__ __forceinline__ void zero_d_pad(uint16_t* d_out, int64_t nb) {
  for (int64_t i = nb; i % 8 != 0; ++i) d_out[i] = 0;
}

__global__ void q4_0_kernel(const float* __restrict__ W, int64_t nb, uint8_t* __restrict__ packed,
                            uint16_t* __restrict__ d_out) {
  const int64_t b = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (b == 0) zero_d_pad(d_out, nb);
  if (b >= nb) return;
  const float4* src = reinterpret_cast<const float4*>(W + b * kGGBlock);
  float v[kGGBlock];
#pragma unroll
  for (int i = 0; i < kGGBlock / 4; ++i) {
    const float4 t = src[i];
    v[4 * i] = t.x; v[4 * i + 1] = t.y; v[4 * i + 2] = t.z; v[4 * i + 3] = t.w;
  }
  float best = -1.0f, ext = 0.0f;
#pragma unroll
  for (int i = 0; i < kGGBlock; ++i)
    if (fabsf(v[i]) > best) { best = fabsf(v[i]); ext = v[i]; }  // strict: first index wins ties
  const __half d16 = __float2half_rn(__fdiv_rn(ext, -8.0f));
  const float d = __half2float(d16);
  uint32_t w[4] = {0, 0, 0, 0};
#pragma unroll
  for (int i = 0; i < kGGBlock; ++i) {
    float q = 8.0f;
    if (d != 0.0f) q = fminf(fmaxf(__fadd_rn(rintf(__fdiv_rn(v[i], d)), 8.0f), 0.0f), 15.0f);
    w[i >> 3] |= ((uint32_t)q) << (4 * (i & 7));
  }
  reinterpret_cast<uint4*>(packed)[b] = make_uint4(w[0], w[1], w[2], w[3]);
  d_out[b] = __half_as_ushort(d16);
}

__global__ void q8_0_kernel(const float* __restrict__ W, int64_t nb, int8_t* __restrict__ packed,
                            uint16_t* __restrict__ d_out) {
  const int64_t b = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (b == 0) zero_d_pad(d_out, nb);
  if (b >= nb) return;
  const float4* src = reinterpret_cast<const float4*>(W + b * kGGBlock);
  float v[kGGBlock];
  float amax = 0.0f;
#pragma unroll
  for (int i = 0; i < kGGBlock / 4; ++i) {
    const float4 t = src[i];
    v[4 * i] = t.x; v[4 * i + 1] = t.y; v[4 * i + 2] = t.z; v[4 * i + 3] = t.w;
    amax = fmaxf(amax, fmaxf(fmaxf(fabsf(t.x), fabsf(t.y)), fmaxf(fabsf(t.z), fabsf(t.w))));
  }
  const __half d16 = __float2half_rn(__fdiv_rn(amax, 127.0f));
  const float d = __half2float(d16);
  uint32_t w[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) w[i] = 0;
#pragma unroll
  for (int i = 0; i < kGGBlock; ++i) {
    float q = 0.0f;
    if (d != 0.0f) q = fminf(fmaxf(rintf(__fdiv_rn(v[i], d)), -127.0f), 127.0f);
    w[i >> 2] |= ((uint32_t)(uint8_t)(int8_t)(int)q) << (8 * (i & 3));
  }
  uint4* dst = reinterpret_cast<uint4*>(packed + b * kGGBlock);
  dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
  dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
  d_out[b] = __half_as_ushort(d16);
}

// q4_1: m = fp16(min), d = fp16((max - min) / 15), q = clamp(rint((x - m) / d), 0, 15) against the
// stored m and d (q = 0 where d == 0).  Storage unit of 128 elements: 64 bytes of nibbles, then the
// four blocks' (d, m) fp16 pairs; block b of a unit owns nibble bytes [16b, 16b + 16) and pair
// bytes [64 + 4b, 64 + 4b + 4).  The scales blob is 16 zero bytes.
__global__ void q4_1_kernel(const float* __restrict__ W, int64_t nb, uint8_t* __restrict__ packed,
                            uint32_t* __restrict__ scales) {
  const int64_t b = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (b == 0)
    for (int i = 0; i < 4; ++i) scales[i] = 0u;
  if (b >= nb) return;
  const float4* src = reinterpret_cast<const float4*>(W + b * kGGBlock);
  float v[kGGBlock];
  float mn = INFINITY, mx = -INFINITY;
#pragma unroll
  for (int i = 0; i < kGGBlock / 4; ++i) {
    const float4 t = src[i];
    v[4 * i] = t.x; v[4 * i + 1] = t.y; v[4 * i + 2] = t.z; v[4 * i + 3] = t.w;
  }
#pragma unroll
  for (int i = 0; i < kGGBlock; ++i) { mn = fminf(mn, v[i]); mx = fmaxf(mx, v[i]); }
  const __half d16 = __float2half_rn(__fdiv_rn(__fsub_rn(mx, mn), 15.0f));
  const __half m16 = __float2half_rn(mn);
  const float d = __half2float(d16), m = __half2float(m16);
  uint32_t w[4] = {0, 0, 0, 0};
#pragma unroll
  for (int i = 0; i < kGGBlock; ++i) {
    float q = 0.0f;
    if (d != 0.0f) q = fminf(fmaxf(rintf(__fdiv_rn(__fsub_rn(v[i], m), d)), 0.0f), 15.0f);
    w[i >> 3] |= ((uint32_t)q) << (4 * (i & 7));
  }
  uint8_t* unit = packed + (b / 4) * 80;
  *reinterpret_cast<uint4*>(unit + 16 * (b % 4)) = make_uint4(w[0], w[1], w[2], w[3]);
  *reinterpret_cast<uint32_t*>(unit + 64 + 4 * (b % 4)) =
      (uint32_t)__half_as_ushort(d16) | ((uint32_t)__half_as_ushort(m16) << 16);
}

// q5_0: d = fp16(extreme / -16), q = clamp(rint(x / d) + 16, 0, 31) (q = 16 where d == 0).  Storage
// unit of 128 elements: 64 bytes of low nibbles, then 16 bytes of fifth bits; block b of a unit owns
// nibble bytes [16b, 16b + 16) and fifth-bit bytes [64 + 4b, 64 + 4b + 4).
__global__ void q5_0_kernel(const float* __restrict__ W, int64_t nb, uint8_t* __restrict__ packed,
                            uint16_t* __restrict__ d_out) {
  const int64_t b = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (b == 0) zero_d_pad(d_out, nb);
  if (b >= nb) return;
  const float4* src = reinterpret_cast<const float4*>(W + b * kGGBlock);
  float v[kGGBlock];
#pragma unroll
  for (int i = 0; i < kGGBlock / 4; ++i) {
    const float4 t = src[i];
    v[4 * i] = t.x; v[4 * i + 1] = t.y; v[4 * i + 2] = t.z; v[4 * i + 3] = t.w;
  }
  float best = -1.0f, ext = 0.0f;
#pragma unroll
  for (int i = 0; i < kGGBlock; ++i)
    if (fabsf(v[i]) > best) { best = fabsf(v[i]); ext = v[i]; }  // strict: first index wins ties
  const __half d16 = __float2half_rn(__fdiv_rn(ext, -16.0f));
  const float d = __half2float(d16);
  uint32_t w[4] = {0, 0, 0, 0}, hb = 0;
#pragma unroll
  for (int i = 0; i < kGGBlock; ++i) {
    float q = 16.0f;
    if (d != 0.0f) q = fminf(fmaxf(__fadd_rn(rintf(__fdiv_rn(v[i], d)), 16.0f), 0.0f), 31.0f);
    const uint32_t qi = (uint32_t)q;
    w[i >> 3] |= (qi & 15u) << (4 * (i & 7));
    hb |= (qi >> 4) << i;
  }
  const int64_t unit = b / 4, blk = b % 4;
  uint8_t* base = packed + unit * 80;
  *reinterpret_cast<uint4*>(base + 16 * blk) = make_uint4(w[0], w[1], w[2], w[3]);
  *reinterpret_cast<uint32_t*>(base + 64 + 4 * blk) = hb;
  d_out[b] = __half_as_ushort(d16);
}

// FP8 E4M3 weights, one warp per row: s = amax(row) / 448, q = E4M3(w / s) (0 where s == 0).
__global__ void fp8_kernel(const float* __restrict__ W, int64_t N, int64_t K, uint8_t* __restrict__ packed,
                           float* __restrict__ s_out, int pad_words) {
  const int64_t n = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (n == 0 && lane < pad_words) s_out[N + lane] = 0.0f;  // zero the pad to 16 bytes
  if (n >= N) return;
  const float* row = W + n * K;
  float a = 0.0f;
  for (int64_t k = 4 * lane; k < K; k += 128) {
    const float4 t = *reinterpret_cast<const float4*>(row + k);
    a = fmaxf(a, fmaxf(fmaxf(fabsf(t.x), fabsf(t.y)), fmaxf(fabsf(t.z), fabsf(t.w))));
  }
  a = __uint_as_float(__reduce_max_sync(0xFFFFFFFFu, __float_as_uint(a)));
  const float sc = __fdiv_rn(a, 448.0f);
  if (lane == 0) s_out[n] = sc;
  for (int64_t k = 4 * lane; k < K; k += 128) {
    const float4 t = *reinterpret_cast<const float4*>(row + k);
    const float x[4] = {t.x, t.y, t.z, t.w};
    uint32_t w = 0;
#pragma unroll
    for (int j = 0; j < 4; ++j) w |= (sc == 0.0f ? 0u : f32_to_e4m3_satfinite(__fdiv_rn(x[j], sc))) << (8 * j);
    *reinterpret_cast<uint32_t*>(packed + n * K + k) = w;
  }
}

// ------------------------------------------------------------------ dequant export
// one thread per 8 consecutive elements
__global__ void dequant_kernel(const uint8_t* __restrict__ packed, const uint8_t* __restrict__ scales, int fmt,
                               int64_t n8, int64_t K, ScalesLayout lay, float* __restrict__ out) {
  const int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (t >= n8) return;
  const int64_t e0 = t * 8;
  float r[8];
  if (fmt == WQ_FP8) {
    const uint2 c = reinterpret_cast<const uint2*>(packed)[t];
    const float sc = reinterpret_cast<const float*>(scales)[e0 / K];
#pragma unroll
    for (int j = 0; j < 8; ++j) r[j] = __fmul_rn(e4m3_to_f32(((j < 4 ? c.x : c.y) >> (8 * (j & 3))) & 0xFFu), sc);
  } else if (fmt == WQ_Q5_0) {
    const int64_t unit = e0 / 128, off = e0 % 128;
    const uint32_t c = *reinterpret_cast<const uint32_t*>(packed + unit * 80 + off / 2);
    const uint32_t hb = packed[unit * 80 + 64 + off / 8];
    const float d = f16_bits_to_f32(reinterpret_cast<const uint16_t*>(scales)[e0 / kGGBlock]);
#pragma unroll
    for (int j = 0; j < 8; ++j)
      r[j] = __fmul_rn((float)((int)(((c >> (4 * j)) & 15u) | (((hb >> j) & 1u) << 4)) - 16), d);
  } else if (fmt == WQ_Q8_0) {
    const uint2 c = reinterpret_cast<const uint2*>(packed)[t];
    const float d = f16_bits_to_f32(reinterpret_cast<const uint16_t*>(scales)[e0 / kGGBlock]);
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int8_t q = (int8_t)(((j < 4 ? c.x : c.y) >> (8 * (j & 3))) & 0xFF);
      r[j] = __fmul_rn((float)q, d);
    }
  } else {
    const uint32_t c = (fmt == WQ_Q4_1)
                           ? *reinterpret_cast<const uint32_t*>(packed + (e0 / 128) * 80 + (e0 % 128) / 2)
                           : reinterpret_cast<const uint32_t*>(packed)[t];
    if (fmt == WQ_NF4) {
      const int64_t b = e0 / kNF4Block;
      const int8_t q = reinterpret_cast<const int8_t*>(scales)[b];
      const float s2 = reinterpret_cast<const float*>(scales + lay.s2_off)[b / kDQGroup];
      const float off = *reinterpret_cast<const float*>(scales + lay.offset_off);
      const float a = __fadd_rn(__fmul_rn((float)q, s2), off);
#pragma unroll
      for (int j = 0; j < 8; ++j) r[j] = __fmul_rn(kNF4[(c >> (4 * j)) & 15u], a);
    } else if (fmt == WQ_NVFP4 || fmt == WQ_NVFP4_W4A4) {
      const float s = e4m3_to_f32(scales[e0 / kNVBlock]);
      const float g = *reinterpret_cast<const float*>(scales + lay.g_off);
#pragma unroll
      for (int j = 0; j < 8; ++j) r[j] = __fmul_rn(__fmul_rn(kE2M1[(c >> (4 * j)) & 15u], s), g);
    } else if (fmt == WQ_Q4_1) {
      const uint32_t dm = *reinterpret_cast<const uint32_t*>(packed + (e0 / 128) * 80 + 64 + 4 * ((e0 % 128) / 32));
      const float d = f16_bits_to_f32(dm & 0xFFFFu), m = f16_bits_to_f32(dm >> 16);
#pragma unroll
      for (int j = 0; j < 8; ++j) r[j] = __fadd_rn(__fmul_rn((float)((c >> (4 * j)) & 15u), d), m);
    } else {  // q4_0
      const float d = f16_bits_to_f32(reinterpret_cast<const uint16_t*>(scales)[e0 / kGGBlock]);
#pragma unroll
      for (int j = 0; j < 8; ++j) r[j] = __fmul_rn((float)((int)((c >> (4 * j)) & 15u) - 8), d);
    }
  }
  float4* o = reinterpret_cast<float4*>(out + e0);
  o[0] = make_float4(r[0], r[1], r[2], r[3]);
  o[1] = make_float4(r[4], r[5], r[6], r[7]);
}

inline int launch_status() {
  cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? WQ_OK : WQ_ERR_CUDA;
}

}  // namespace

// ------------------------------------------------------------------ host entry points
int pack_nf4(const float* W, int64_t N, int64_t K, uint8_t* packed, uint8_t* scales, cudaStream_t s) {
  const int64_t nb = N * K / kNF4Block;
  if (nb == 0) return WQ_OK;
  const ScalesLayout lay = scales_layout(WQ_NF4, N, K);
  // the packed output (32 bytes per block) holds the fp32 absmax values and the exponent buckets
  // until the codes kernel, the last one, overwrites it
  float* tmp = reinterpret_cast<float*>(packed);
  const int64_t bucket_off = (nb * 4 + 7) / 8 * 8;
  int8_t* absmax_q = reinterpret_cast<int8_t*>(scales);
  float* s2 = reinterpret_cast<float*>(scales + lay.s2_off);
  float* offset = reinterpret_cast<float*>(scales + lay.offset_off);
  nf4_absmax_kernel<<<grid_for(nb, 256), 256, 0, s>>>(W, nb, tmp);
  // one CTA is quicker below ~16 K blocks (a 384 x 1536 weight: 42 against 50 us on GB300); above
  // that the parallel form wins (5120 x 1280: 70 against 167 us)
  if (nb >= 16384 && bucket_off + 256 * 8 <= nb * (kNF4Block / 2)) {
    auto* gbucket = reinterpret_cast<unsigned long long*>(packed + bucket_off);
    if (cudaMemsetAsync(gbucket, 0, 256 * 8, s) != cudaSuccess) return WQ_ERR_CUDA;
    int g = grid_for(nb, 1024);
    if (g > 152) g = 152;
    nf4_bucket_kernel<<<g, 1024, 0, s>>>(tmp, nb, gbucket);
    nf4_offset_kernel<<<1, 256, 0, s>>>(gbucket, nb, offset, absmax_q, (int64_t)lay.s2_off);
    nf4_dq_groups_kernel<<<grid_for((nb + kDQGroup - 1) / kDQGroup * 32, 256), 256, 0, s>>>(tmp, nb, offset,
                                                                                          absmax_q, s2);
    count_launch(3);
  } else {  // small weights: one CTA
    nf4_double_quant_kernel<<<1, 1024, 0, s>>>(tmp, nb, absmax_q, s2, offset, (int64_t)lay.s2_off);
    count_launch();
  }
  nf4_codes_kernel<<<grid_for(nb, 128), 128, 0, s>>>(W, nb, packed);
  count_launch(2);
  return launch_status();
}

int pack_nvfp4(const float* W, int64_t N, int64_t K, uint8_t* packed, uint8_t* scales, cudaStream_t s) {
  const int64_t n = N * K, nblk = n / kNVBlock;
  if (n == 0) return WQ_OK;
  const ScalesLayout lay = scales_layout(WQ_NVFP4, N, K);
  float* slot = reinterpret_cast<float*>(scales + lay.g_off);
  if (cudaMemsetAsync(slot, 0, sizeof(float), s) != cudaSuccess) return WQ_ERR_CUDA;
  int g = grid_for(n / 8, 256);
  if (g > 304) g = 304;  // about two blocks per SM, each looping; one atomic per block
  amax_kernel<float><<<g, 256, 0, s>>>(W, n, reinterpret_cast<unsigned*>(slot));
  nvfp4_quant_kernel<float><<<grid_for(nblk, 256), 256, 0, s>>>(W, nblk, slot, 1, packed, scales, nullptr);
  nvfp4_finalize_kernel<<<1, 32, 0, s>>>(slot, scales + lay.sf_bytes, (int)(lay.g_off - lay.sf_bytes));
  count_launch(3);
  return launch_status();
}

int pack_q4_0(const float* W, int64_t N, int64_t K, uint8_t* packed, uint8_t* scales, cudaStream_t s) {
  const int64_t nb = N * K / kGGBlock;
  if (nb == 0) return WQ_OK;
  q4_0_kernel<<<grid_for(nb, 128), 128, 0, s>>>(W, nb, packed, reinterpret_cast<uint16_t*>(scales));
  count_launch();
  return launch_status();
}

int pack_q8_0(const float* W, int64_t N, int64_t K, uint8_t* packed, uint8_t* scales, cudaStream_t s) {
  const int64_t nb = N * K / kGGBlock;
  if (nb == 0) return WQ_OK;
  q8_0_kernel<<<grid_for(nb, 128), 128, 0, s>>>(W, nb, reinterpret_cast<int8_t*>(packed),
                                                reinterpret_cast<uint16_t*>(scales));
  count_launch();
  return launch_status();
}

int pack_q4_1(const float* W, int64_t N, int64_t K, uint8_t* packed, uint8_t* scales, cudaStream_t s) {
  const int64_t nb = N * K / kGGBlock;
  if (nb == 0) return WQ_OK;
  q4_1_kernel<<<grid_for(nb, 128), 128, 0, s>>>(W, nb, packed, reinterpret_cast<uint32_t*>(scales));
  count_launch();
  return launch_status();
}

int pack_q5_0(const float* W, int64_t N, int64_t K, uint8_t* packed, uint8_t* scales, cudaStream_t s) {
  const int64_t nb = N * K / kGGBlock;
  if (nb == 0) return WQ_OK;
  q5_0_kernel<<<grid_for(nb, 128), 128, 0, s>>>(W, nb, packed, reinterpret_cast<uint16_t*>(scales));
  count_launch();
  return launch_status();
}

int pack_fp8(const float* W, int64_t N, int64_t K, uint8_t* packed, uint8_t* scales, cudaStream_t s) {
  if (N * K == 0) return WQ_OK;
  const int pad_words = (int)((align16((size_t)N * 4) - (size_t)N * 4) / 4);
  fp8_kernel<<<grid_for(N, 8), 256, 0, s>>>(W, N, K, packed, reinterpret_cast<float*>(scales), pad_words);
  count_launch();
  return launch_status();
}

int dequant(const uint8_t* packed, const uint8_t* scales, int fmt, int64_t N, int64_t K, float* out,
            cudaStream_t s) {
  const int64_t n8 = N * K / 8;
  if (n8 == 0) return WQ_OK;
  dequant_kernel<<<grid_for(n8, 256), 256, 0, s>>>(packed, scales, fmt, n8, K, scales_layout(fmt, N, K), out);
  count_launch();
  return launch_status();
}

// Failure-path self test: one thread waits on an mbarrier that nothing arrives on, with the
// same bounded poll the pipelines use, and records WQ_STATUS_TIMEOUT once it gives up.
__global__ void selftest_timeout_kernel(uint32_t polls) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    uint32_t i = 0;
    while (i < polls && !mbar_try_wait(&bar, 0)) ++i;
    if (i == polls) set_status(WQ_STATUS_TIMEOUT);
  }
}

// Scalar-encoder self test: for each fp32 input, the library's own E2M1 and E4M3 encoders
// (the ones the packers and the activation quantiser use) next to the hardware conversions
// cvt.rn.satfinite.{e2m1x2,e4m3x2}.f32 on the same value, so a test can compare both with
// the oracle (ties, signed zeros, subnormal and saturating scales).
__global__ void selftest_encoders_kernel(const float* __restrict__ in, int64_t n, uint8_t* __restrict__ out) {
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n) return;
  const float x = in[i];
  uint32_t hw_e2m1, hw_e4m3;
  // the converted value of the first source lands in the upper half, the second in the lower
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b0, %1, %2;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b1, %1, %1;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b2, %1, %1;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b3, %1, %1;\n\t"
      "mov.b32 %0, {b0, b1, b2, b3};\n\t}"
      : "=r"(hw_e2m1)
      : "f"(0.0f), "f"(x));
  uint16_t h;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(h) : "f"(0.0f), "f"(x));
  hw_e4m3 = h & 0xFFu;
  out[4 * i + 0] = (uint8_t)f32_to_e2m1(x);
  out[4 * i + 1] = (uint8_t)(hw_e2m1 & 0xFu);
  out[4 * i + 2] = (uint8_t)f32_to_e4m3_satfinite(x);
  out[4 * i + 3] = (uint8_t)hw_e4m3;
}

int selftest_encoders(const float* in, int64_t n, uint8_t* out, cudaStream_t s) {
  if (n == 0) return WQ_OK;
  selftest_encoders_kernel<<<grid_for(n, 256), 256, 0, s>>>(in, n, out);
  count_launch();
  return launch_status();
}

int selftest_timeout(uint32_t polls, cudaStream_t s) {
  selftest_timeout_kernel<<<1, 32, 0, s>>>(polls);
  count_launch();
  return launch_status();
}

static int sm_count() {
  static int n = 0;
  static std::once_flag once;
  std::call_once(once, [] {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n < 1)
      n = 148;
  });
  return n;
}

int quant_act_nvfp4(const uint16_t* x, int64_t M, int64_t K, const float* g_in, uint8_t* codes,
                    uint8_t* scales, float* g_out, cudaStream_t s) {
  const int64_t n = M * K, nblk = n / kNVBlock;
  if (n == 0) return WQ_OK;
  if (g_in) {
    nvfp4_quant_kernel<uint16_t><<<grid_for(nblk, 256), 256, 0, s>>>(x, nblk, g_in, 0, codes, scales, g_out);
    count_launch();
    return launch_status();
  }
  if (cudaMemsetAsync(g_out, 0, sizeof(float), s) != cudaSuccess) return WQ_ERR_CUDA;
  // four CTAs per SM, each thread with four 16-byte loads in flight
  int g = grid_for(n / 8, 256);
  if (g > 4 * sm_count()) g = 4 * sm_count();
  amax_kernel<uint16_t><<<g, 256, 0, s>>>(x, n, reinterpret_cast<unsigned*>(g_out));
  // the quantiser and the finalisation start while their predecessor finishes (programmatic
  // dependent launch); each waits for it before reading the amax slot
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid_for(nblk, 256));
  cfg.blockDim = dim3(256);
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, nvfp4_quant_kernel<uint16_t>, x, nblk, (const float*)g_out, 1, codes, scales,
                         (float*)nullptr) != cudaSuccess)
    return WQ_ERR_CUDA;
  cfg.gridDim = dim3(1);
  cfg.blockDim = dim3(32);
  if (cudaLaunchKernelEx(&cfg, nvfp4_finalize_kernel, g_out, (uint8_t*)nullptr, 0) != cudaSuccess) return WQ_ERR_CUDA;
  count_launch(3);
  return launch_status();
}

int take_status_pack() {
  int v = 0, zero = 0;
  if (cudaMemcpyFromSymbol(&v, g_status, sizeof(int)) != cudaSuccess) return WQ_ERR_CUDA;
  cudaMemcpyToSymbol(g_status, &zero, sizeof(int));
  return v;
}

}  // namespace wq
