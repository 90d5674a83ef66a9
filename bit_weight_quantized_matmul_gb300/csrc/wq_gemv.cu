// wq_gemv.cu -- one Linear at decode sizes (M <= 16 activation rows) on the CUDA cores.
//
// The per-token decode step runs each Linear as its own launch (PR "Run quantized Whisper on
// the fused Metal decode path", "Summary": a quantized single-row kernel; "Measurements": at
// these sizes per-token decode is bound by dispatch, not by weight bandwidth).  A 1280 x 1280 NF4
// weight is 0.85 MB, a fraction of a microsecond of HBM time, so what the kernel must minimise is
// latency: every weight load of a thread is issued at once, before the kernel waits for the
// preceding one (programmatic dependent launch: weights, scales and bias do not depend on it), the
// activations arrive with one round of asynchronous copies, and no tensor-memory, barrier-ring or
// cluster set-up is paid.  Work per weight is ~M multiply-adds, small enough for the CUDA cores
// (packed fp32x2 FMAs).
//
// Mapping: a CTA of kWarps warps owns kWarps * kR consecutive weight rows; in a warp, lane l
// holds the 32-element pieces l, l + 32, ... of each of its kR rows.  Weights are decoded to the
// exact fp32 value wq_dequant gives and multiplied with x (bf16 -> fp32) in fp32; the lanes'
// partial sums are added with warp shuffles.  Formats: every weight format of the library.
#include <cuda_runtime.h>

#include <mutex>

#include "wq_device.cuh"
#include "wq_internal.h"

namespace wq {
namespace {

constexpr int kWarps = 4;          // warps per CTA
constexpr int kR = 2;              // weight rows per warp
constexpr int kPLMax = 5;          // 32-element pieces per lane: K <= 32 * 32 * 5 = 5120
constexpr int kXSmemMax = 160 * 1024;  // activation bytes staged per CTA (M * K * 2)

struct GemvParams {
  const uint16_t* x;
  const uint8_t* packed;
  const uint8_t* scales;
  const uint16_t* bias;
  int M, N, K;
  int out_f32;
  uint32_t s2_off, offset_off, g_off;
  void* ys[WQ_OUT_MAX];
  int ld[WQ_OUT_MAX];
  int col_end[WQ_OUT_MAX];
};

template <int FMT>
struct GFmt {
  static constexpr bool BYTE = FMT == WQ_Q8_0 || FMT == WQ_FP8;
  static constexpr int PW = BYTE ? 2 : 1;  // 16-byte words of codes per 32-element piece
};

__device__ __forceinline__ uint4 ld_stream_v4(const uint8_t* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

__device__ __forceinline__ void cp_async16(uint32_t smem_addr, const void* g) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_addr), "l"(g) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

// physical 16-byte slot of activation chunk c in shared memory: the two low bits are XOR-ed with
// bits 3-4, so the 8 lanes of one phase of a 16-byte load (chunks 4l + i, l = 0..7) hit 8 different
// bank groups
__device__ __forceinline__ int xslot(int c) { return c ^ ((c >> 3) & 3); }

// Exact fp32 value of code table entry i (the 4-bit codebook formats and q5_0).
template <int FMT>
__device__ __forceinline__ float code_value(int i) {
  if (FMT == WQ_NF4) return kNF4[i & 15];
  if (FMT == WQ_NVFP4) return kE2M1[i & 15];
  if (FMT == WQ_Q4_0) return (float)((i & 15) - 8);
  if (FMT == WQ_Q4_1) return (float)(i & 15);
  if (FMT == WQ_Q5_0) return (float)((i & 31) - 16);
  return 0.0f;
}

template <int FMT, int MT>
__global__ void __launch_bounds__(kWarps * 32) wq_gemv_kernel(GemvParams p) {
  extern __shared__ __align__(16) uint8_t xs_raw[];
  __shared__ float tab[32];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int npieces = p.K / 32;
  const int64_t row0 = ((int64_t)blockIdx.x * kWarps + warp) * kR;

  // ---- weights, scales and bias of this lane's pieces: every load issued before any is used
  uint4 wv[kR][kPLMax][GFmt<FMT>::PW];
  uint32_t sw[kR][kPLMax];   // raw scale word of each piece (format-specific)
  float s2v[kR][kPLMax];     // NF4: second-level scale of the piece's block
  uint32_t hb[kR][kPLMax];   // q5_0: the piece's fifth bits; q4_1: its (d, m) pair
#pragma unroll
  for (int r = 0; r < kR; ++r) {
    const int64_t n = row0 + r;
    const bool row_ok = n < p.N;
#pragma unroll
    for (int j = 0; j < kPLMax; ++j) {
      const int pc = lane + 32 * j;
      sw[r][j] = 0u;
      s2v[r][j] = 0.0f;
      hb[r][j] = 0u;
#pragma unroll
      for (int w = 0; w < GFmt<FMT>::PW; ++w) wv[r][j][w] = make_uint4(0u, 0u, 0u, 0u);
      if (!row_ok || pc >= npieces) continue;
      const int64_t e0 = n * p.K + (int64_t)pc * 32;  // first element of the piece
      if (FMT == WQ_Q5_0 || FMT == WQ_Q4_1) {  // 80-byte unit: nibbles, then side data per block
        const uint8_t* unit = p.packed + (e0 / 128) * 80;
        wv[r][j][0] = ld_stream_v4(unit + (pc & 3) * 16);
        hb[r][j] = __ldg(reinterpret_cast<const uint32_t*>(unit + 64) + (pc & 3));
      } else if (GFmt<FMT>::BYTE) {
        wv[r][j][0] = ld_stream_v4(p.packed + e0);
        wv[r][j][1] = ld_stream_v4(p.packed + e0 + 16);
      } else {
        wv[r][j][0] = ld_stream_v4(p.packed + e0 / 2);
      }
      if (FMT == WQ_NF4) {
        const int64_t b = e0 / 64;
        sw[r][j] = (uint32_t)(uint8_t)__ldg(reinterpret_cast<const int8_t*>(p.scales) + b);
        s2v[r][j] = __ldg(reinterpret_cast<const float*>(p.scales + p.s2_off) + b / 256);
      } else if (FMT == WQ_NVFP4) {
        sw[r][j] = __ldg(reinterpret_cast<const uint16_t*>(p.scales) + e0 / 32);  // two E4M3 bytes
      } else if (FMT == WQ_Q4_1) {
        // (d, m) read with the codes above
      } else if (FMT == WQ_FP8) {
        if (j == 0) sw[r][0] = __float_as_uint(__ldg(reinterpret_cast<const float*>(p.scales) + n));
      } else {
        sw[r][j] = __ldg(reinterpret_cast<const uint16_t*>(p.scales) + e0 / 32);  // fp16 d
      }
    }
  }
  float off = 0.0f, gsc = 1.0f;
  if (FMT == WQ_NF4) off = __ldg(reinterpret_cast<const float*>(p.scales + p.offset_off));
  if (FMT == WQ_NVFP4) gsc = __ldg(reinterpret_cast<const float*>(p.scales + p.g_off));
  float bias_r[kR];
#pragma unroll
  for (int r = 0; r < kR; ++r)
    bias_r[r] = (p.bias && row0 + r < p.N) ? bf16_bits_to_f32(__ldg(p.bias + row0 + r)) : 0.0f;
  if (threadIdx.x < 32) tab[threadIdx.x] = code_value<FMT>(threadIdx.x);
  griddep_launch_dependents();

  // ---- activations: wait for the preceding kernel, then one round of asynchronous 16-byte copies
  griddep_wait();
  const int nchunk = p.M * p.K / 8;
  const uint32_t xs = smem_u32(xs_raw);
  for (int c = threadIdx.x; c < nchunk; c += kWarps * 32)
    cp_async16(xs + 16u * (uint32_t)xslot(c), p.x + (int64_t)c * 8);
  cp_async_wait_all();
  __syncthreads();

  // ---- decode and multiply
  float2 acc[kR][MT];
#pragma unroll
  for (int r = 0; r < kR; ++r)
#pragma unroll
    for (int m = 0; m < MT; ++m) acc[r][m] = make_float2(0.0f, 0.0f);
#pragma unroll
  for (int j = 0; j < kPLMax; ++j) {
    const int pc = lane + 32 * j;
    if (pc >= npieces) break;
    float w[kR][32];
#pragma unroll
    for (int r = 0; r < kR; ++r) {
      if (GFmt<FMT>::BYTE) {
        const float sc = (FMT == WQ_FP8) ? __uint_as_float(sw[r][0]) : f16_bits_to_f32(sw[r][j]);
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const uint32_t u[4] = {wv[r][j][h].x, wv[r][j][h].y, wv[r][j][h].z, wv[r][j][h].w};
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            const uint32_t byte = (u[e >> 2] >> (8 * (e & 3))) & 0xFFu;
            const float v = (FMT == WQ_FP8) ? e4m3_to_f32(byte) : (float)(int8_t)byte;
            w[r][h * 16 + e] = __fmul_rn(v, sc);
          }
        }
      } else {
        const uint32_t u[4] = {wv[r][j][0].x, wv[r][j][0].y, wv[r][j][0].z, wv[r][j][0].w};
        float sa = 0.0f, sb = 0.0f, madd = 0.0f;  // scale of elements 0..15 and 16..31, q4_1 minimum
        if (FMT == WQ_NF4) {
          sa = sb = __fadd_rn(__fmul_rn((float)(int8_t)sw[r][j], s2v[r][j]), off);
        } else if (FMT == WQ_NVFP4) {
          sa = e4m3_to_f32(sw[r][j] & 0xFFu);
          sb = e4m3_to_f32(sw[r][j] >> 8);
        } else if (FMT == WQ_Q4_1) {
          sa = sb = f16_bits_to_f32(hb[r][j] & 0xFFFFu);
          madd = f16_bits_to_f32(hb[r][j] >> 16);
        } else {
          sa = sb = f16_bits_to_f32(sw[r][j]);
        }
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          uint32_t code = (u[e >> 3] >> (4 * (e & 7))) & 15u;
          if (FMT == WQ_Q5_0) code |= ((hb[r][j] >> e) & 1u) << 4;
          const float s = e < 16 ? sa : sb;
          float v = __fmul_rn(tab[code], s);
          if (FMT == WQ_NVFP4) v = __fmul_rn(v, gsc);
          if (FMT == WQ_Q4_1) v = __fadd_rn(v, madd);
          w[r][e] = v;
        }
      }
    }
#pragma unroll
    for (int m = 0; m < MT; ++m) {
      if (m >= p.M) break;
      const int c0 = m * (p.K / 8) + pc * 4;  // first 16-byte chunk of x[m, piece]
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const uint4 xv = *reinterpret_cast<const uint4*>(xs_raw + 16 * xslot(c0 + i));
        const uint32_t xw[4] = {xv.x, xv.y, xv.z, xv.w};
#pragma unroll
        for (int t = 0; t < 4; ++t) {
          const float2 x2 = make_float2(__uint_as_float(xw[t] << 16), __uint_as_float(xw[t] & 0xFFFF0000u));
#pragma unroll
          for (int r = 0; r < kR; ++r)
            acc[r][m] = __ffma2_rn(make_float2(w[r][i * 8 + 2 * t], w[r][i * 8 + 2 * t + 1]), x2, acc[r][m]);
        }
      }
    }
  }

  // ---- reduce over the lanes, add the bias, store
#pragma unroll
  for (int r = 0; r < kR; ++r) {
#pragma unroll
    for (int m = 0; m < MT; ++m) {
      float v = acc[r][m].x + acc[r][m].y;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
      const int64_t n = row0 + r;
      if (lane == ((r * MT + m) & 31) && m < p.M && n < p.N) {
        int d = 0;
#pragma unroll
        for (int i = 0; i < WQ_OUT_MAX - 1; ++i) d += (n >= p.col_end[i]) ? 1 : 0;
        const int64_t at = (int64_t)m * p.ld[d] + (n - (d ? p.col_end[d - 1] : 0));
        const float val = __fadd_rn(v, bias_r[r]);
        if (p.out_f32)
          reinterpret_cast<float*>(p.ys[d])[at] = val;
        else
          reinterpret_cast<__nv_bfloat16*>(p.ys[d])[at] = __float2bfloat16_rn(val);
      }
    }
  }
}

template <int FMT, int MT>
int launch_gemv(const LinearArgs& a, cudaStream_t s) {
  auto kern = wq_gemv_kernel<FMT, MT>;
  static std::once_flag once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(once, [&] {
    attr_err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kXSmemMax);
  });
  if (attr_err != cudaSuccess) return WQ_ERR_CUDA;
  GemvParams p{};
  p.x = reinterpret_cast<const uint16_t*>(a.x);
  p.packed = a.packed;
  p.scales = a.scales;
  p.bias = a.bias;
  p.M = (int)a.M;
  p.N = (int)a.N;
  p.K = (int)a.K;
  p.out_f32 = a.out_f32 ? 1 : 0;
  const ScalesLayout L = scales_layout(FMT, a.N, a.K);
  p.s2_off = (uint32_t)L.s2_off;
  p.offset_off = (uint32_t)L.offset_off;
  p.g_off = (uint32_t)L.g_off;
  for (int d = 0; d < WQ_OUT_MAX; ++d) {
    const int dd = d < a.nout ? d : a.nout - 1;
    p.ys[d] = a.ys[dd];
    p.ld[d] = (int)a.ld[dd];
    p.col_end[d] = (int)a.col_end[dd];
  }
  cudaLaunchConfig_t cfg = {};
  const int rows_per_cta = kWarps * kR;
  cfg.gridDim = dim3((unsigned)((a.N + rows_per_cta - 1) / rows_per_cta), 1, 1);
  cfg.blockDim = dim3(kWarps * 32, 1, 1);
  cfg.dynamicSmemBytes = (size_t)(a.M * a.K * 2);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  cfg.numAttrs = 0;
  if (a.weights_static) {
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
  }
  const cudaError_t e = cudaLaunchKernelEx(&cfg, kern, p);
  count_launch();
  return e == cudaSuccess ? WQ_OK : WQ_ERR_CUDA;
}

template <int FMT>
int dispatch_m(const LinearArgs& a, cudaStream_t s) {
  if (a.M <= 1) return launch_gemv<FMT, 1>(a, s);
  if (a.M <= 2) return launch_gemv<FMT, 2>(a, s);
  if (a.M <= 4) return launch_gemv<FMT, 4>(a, s);
  if (a.M <= 8) return launch_gemv<FMT, 8>(a, s);
  return launch_gemv<FMT, 16>(a, s);
}

}  // namespace

bool gemv_eligible(const LinearArgs& a) {
  if (a.fmt == WQ_NVFP4_W4A4 || a.M < 1 || a.M > 16) return false;
  if (a.K % 32 != 0 || a.K > 32 * 32 * kPLMax) return false;
  if (a.M * a.K * 2 > kXSmemMax) return false;
  if (a.N > 0x7FFFFFFF || ((uintptr_t)a.x & 15u) != 0) return false;
  for (int d = 0; d < a.nout; ++d)
    if (a.ld[d] > 0x7FFFFFFF) return false;
  return true;
}

int linear_gemv(const LinearArgs& a, cudaStream_t s) {
  switch (a.fmt) {
    case WQ_NF4: return dispatch_m<WQ_NF4>(a, s);
    case WQ_NVFP4: return dispatch_m<WQ_NVFP4>(a, s);
    case WQ_Q4_0: return dispatch_m<WQ_Q4_0>(a, s);
    case WQ_Q8_0: return dispatch_m<WQ_Q8_0>(a, s);
    case WQ_Q4_1: return dispatch_m<WQ_Q4_1>(a, s);
    case WQ_Q5_0: return dispatch_m<WQ_Q5_0>(a, s);
    case WQ_FP8: return dispatch_m<WQ_FP8>(a, s);
    default: return WQ_ERR_FMT;
  }
}

}  // namespace wq
