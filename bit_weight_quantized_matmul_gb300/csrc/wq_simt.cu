// wq_simt.cu -- CUDA-core path of y = x . dequant(W)^T (+ bias) for any shape.
//
// Runs where the tensor-core paths' size rules do not hold (and on request).
// Each weight is decoded to its exact fp32 value (the same value wq_dequant
// writes), multiplied in fp32 and reduced across a warp.  W4A4 activations are
// decoded to fp32 the same way.  Source: PR "asr: add a 4-bit nf4 option for
// the Whisper engine", "Why NF4 and not the NVFP4 snapshot" (fused dequant in
// the matmul); model card "whisper-large-v3-turbo -- NVFP4", "What is
// quantized" (W4A4 with runtime activation quantisation).
#include <cuda_runtime.h>

#include "wq_device.cuh"
#include "wq_internal.h"

namespace wq {
namespace {

constexpr int kMT = 8;  // activation rows per pass

struct SimtParams {
  const uint16_t* x;
  const uint8_t* act_codes;
  const uint8_t* act_scales;
  const float* act_g;
  const uint8_t* packed;
  const uint8_t* scales;
  ScalesLayout lay;
  int fmt;
  int64_t M, N, K;
  const uint16_t* bias;
  void* ys[WQ_OUT_MAX];     // columns [col_end[d-1], col_end[d]) of row m at ys[d] + m * ld[d] + (n - col_end[d-1])
  int64_t ld[WQ_OUT_MAX];
  int64_t col_end[WQ_OUT_MAX];
  int out_f32;
};

// 8 consecutive weights of row n starting at column k (k % 8 == 0), exact fp32
__device__ __forceinline__ void decode8(const SimtParams& p, int64_t n, int64_t k, float (&w)[8]) {
  const int64_t e0 = n * p.K + k;
  if (p.fmt == WQ_FP8) {
    const uint2 c = *reinterpret_cast<const uint2*>(p.packed + e0);
    const float sc = reinterpret_cast<const float*>(p.scales)[n];
#pragma unroll
    for (int j = 0; j < 8; ++j) w[j] = __fmul_rn(e4m3_to_f32(((j < 4 ? c.x : c.y) >> (8 * (j & 3))) & 0xFFu), sc);
    return;
  }
  if (p.fmt == WQ_Q5_0) {
    const int64_t unit = e0 / 128, off = e0 % 128;
    const uint32_t c = *reinterpret_cast<const uint32_t*>(p.packed + unit * 80 + off / 2);
    const uint32_t hb = p.packed[unit * 80 + 64 + off / 8];
    const float d = f16_bits_to_f32(reinterpret_cast<const uint16_t*>(p.scales)[e0 / 32]);
#pragma unroll
    for (int j = 0; j < 8; ++j)
      w[j] = __fmul_rn((float)((int)(((c >> (4 * j)) & 15u) | (((hb >> j) & 1u) << 4)) - 16), d);
    return;
  }
  if (p.fmt == WQ_Q8_0) {
    const uint2 c = *reinterpret_cast<const uint2*>(p.packed + e0);
    const float d = f16_bits_to_f32(reinterpret_cast<const uint16_t*>(p.scales)[e0 / 32]);
#pragma unroll
    for (int j = 0; j < 8; ++j) w[j] = __fmul_rn((float)(int8_t)(((j < 4 ? c.x : c.y) >> (8 * (j & 3))) & 0xFF), d);
    return;
  }
  const uint32_t c = (p.fmt == WQ_Q4_1)
                         ? *reinterpret_cast<const uint32_t*>(p.packed + (e0 / 128) * 80 + (e0 % 128) / 2)
                         : *reinterpret_cast<const uint32_t*>(p.packed + e0 / 2);
  if (p.fmt == WQ_NF4) {
    const int64_t b = e0 / 64;
    const int8_t q = reinterpret_cast<const int8_t*>(p.scales)[b];
    const float s2 = reinterpret_cast<const float*>(p.scales + p.lay.s2_off)[b / 256];
    const float off = *reinterpret_cast<const float*>(p.scales + p.lay.offset_off);
    const float a = __fadd_rn(__fmul_rn((float)q, s2), off);
#pragma unroll
    for (int j = 0; j < 8; ++j) w[j] = __fmul_rn(kNF4[(c >> (4 * j)) & 15u], a);
  } else if (p.fmt == WQ_Q4_1) {
    const uint32_t dm = *reinterpret_cast<const uint32_t*>(p.packed + (e0 / 128) * 80 + 64 + 4 * ((e0 % 128) / 32));
    const float d = f16_bits_to_f32(dm & 0xFFFFu), m = f16_bits_to_f32(dm >> 16);
#pragma unroll
    for (int j = 0; j < 8; ++j) w[j] = __fadd_rn(__fmul_rn((float)((c >> (4 * j)) & 15u), d), m);
  } else if (p.fmt == WQ_Q4_0) {
    const float d = f16_bits_to_f32(reinterpret_cast<const uint16_t*>(p.scales)[e0 / 32]);
#pragma unroll
    for (int j = 0; j < 8; ++j) w[j] = __fmul_rn((float)((int)((c >> (4 * j)) & 15u) - 8), d);
  } else {  // NVFP4 weights (W4A16 and W4A4)
    const float s = e4m3_to_f32(p.scales[e0 / 16]);
    const float g = *reinterpret_cast<const float*>(p.scales + p.lay.g_off);
#pragma unroll
    for (int j = 0; j < 8; ++j) w[j] = __fmul_rn(__fmul_rn(kE2M1[(c >> (4 * j)) & 15u], s), g);
  }
}

__device__ __forceinline__ void load_x8(const SimtParams& p, int64_t m, int64_t k, float (&xv)[8]) {
  if (p.fmt == WQ_NVFP4_W4A4) {
    const int64_t e0 = m * p.K + k;
    const uint32_t c = *reinterpret_cast<const uint32_t*>(p.act_codes + e0 / 2);
    const float s = e4m3_to_f32(p.act_scales[e0 / 16]);
    const float g = *p.act_g;
#pragma unroll
    for (int j = 0; j < 8; ++j) xv[j] = __fmul_rn(__fmul_rn(kE2M1[(c >> (4 * j)) & 15u], s), g);
  } else {
    const uint4 v = *reinterpret_cast<const uint4*>(p.x + m * p.K + k);
    const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      xv[2 * j] = bf16_bits_to_f32(u[j] & 0xFFFFu);
      xv[2 * j + 1] = bf16_bits_to_f32(u[j] >> 16);
    }
  }
}

// grid: (ceil(N / warps), ceil(M / kMT)); one warp per weight row, lanes stride K by 8.
__global__ void __launch_bounds__(256) linear_simt_kernel(SimtParams p) {
  const int warps = blockDim.x >> 5;
  const int64_t n = (int64_t)blockIdx.x * warps + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  const int64_t m0 = (int64_t)blockIdx.y * kMT;
  if (n >= p.N) return;
  float acc[kMT];
#pragma unroll
  for (int i = 0; i < kMT; ++i) acc[i] = 0.0f;
  for (int64_t k = (int64_t)lane * 8; k < p.K; k += 32 * 8) {
    float w[8];
    decode8(p, n, k, w);
#pragma unroll
    for (int i = 0; i < kMT; ++i) {
      if (m0 + i < p.M) {
        float xv[8];
        load_x8(p, m0 + i, k, xv);
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[i] = fmaf(xv[j], w[j], acc[i]);
      }
    }
  }
#pragma unroll
  for (int i = 0; i < kMT; ++i) {
    float v = acc[i];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
    acc[i] = v;
  }
  if (lane == 0) {
    const float b = p.bias ? bf16_bits_to_f32(p.bias[n]) : 0.0f;
    int d = 0;
    while (d + 1 < WQ_OUT_MAX && n >= p.col_end[d]) ++d;
    const int64_t col = n - (d ? p.col_end[d - 1] : 0);
    for (int i = 0; i < kMT && m0 + i < p.M; ++i) {
      const float v = acc[i] + b;
      const int64_t off = (m0 + i) * p.ld[d] + col;
      if (p.out_f32)
        reinterpret_cast<float*>(p.ys[d])[off] = v;
      else
        reinterpret_cast<__nv_bfloat16*>(p.ys[d])[off] = __float2bfloat16_rn(v);
    }
  }
}

}  // namespace

int linear_simt(const LinearArgs& a, cudaStream_t s) {
  if (a.M == 0 || a.N == 0) return WQ_OK;
  SimtParams p;
  p.x = reinterpret_cast<const uint16_t*>(a.x);
  p.act_codes = a.act_codes;
  p.act_scales = a.act_scales;
  p.act_g = a.act_g;
  p.packed = a.packed;
  p.scales = a.scales;
  p.lay = scales_layout(a.fmt, a.N, a.K);
  p.fmt = a.fmt;
  p.M = a.M;
  p.N = a.N;
  p.K = a.K;
  p.bias = a.bias;
  for (int d = 0; d < WQ_OUT_MAX; ++d) {
    const int dd = d < a.nout ? d : a.nout - 1;
    p.ys[d] = a.ys[dd];
    p.ld[d] = a.ld[dd];
    p.col_end[d] = a.col_end[dd];
  }
  p.out_f32 = a.out_f32 ? 1 : 0;
  const int warps = 8;
  dim3 grid((unsigned)((a.N + warps - 1) / warps), (unsigned)((a.M + kMT - 1) / kMT));
  if (grid.y > 65535u) return WQ_ERR_SHAPE;
  linear_simt_kernel<<<grid, warps * 32, 0, s>>>(p);
  count_launch();
  return cudaGetLastError() == cudaSuccess ? WQ_OK : WQ_ERR_CUDA;
}

int take_status_simt() {
  int v = 0, zero = 0;
  if (cudaMemcpyFromSymbol(&v, g_status, sizeof(int)) != cudaSuccess) return WQ_ERR_CUDA;
  cudaMemcpyToSymbol(g_status, &zero, sizeof(int));
  return v;
}

}  // namespace wq
