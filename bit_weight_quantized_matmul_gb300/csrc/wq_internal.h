// wq_internal.h -- host-side interfaces between the library's translation units.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/wq.h"

namespace wq {

// Layout of a packed weight's `scales` blob (see include/wq.h).
struct ScalesLayout {
  size_t absmax_bytes = 0;  // NF4: int8 absmax codes
  size_t s2_off = 0;        // NF4: byte offset of the fp32 s2 array
  int64_t n_groups = 0;     // NF4: number of s2 values
  size_t offset_off = 0;    // NF4: byte offset of the fp32 offset
  size_t sf_bytes = 0;      // NVFP4: E4M3 block scales
  size_t g_off = 0;         // NVFP4: byte offset of the fp32 g
  size_t total = 0;
};
// Packed bytes of one weight row (K elements) of a format.
inline int64_t packed_row_bytes(int fmt, int64_t K) {
  switch (fmt) {
    case WQ_Q8_0:
    case WQ_FP8: return K;
    case WQ_Q5_0:
    case WQ_Q4_1: return K / 128 * 80;
    default: return K / 2;
  }
}
ScalesLayout scales_layout(int fmt, int64_t N, int64_t K);

inline size_t align16(size_t n) { return (n + 15) / 16 * 16; }

// Host-side launch counter (all translation units).
void count_launch(int n = 1);

// ---- pack / dequant / activation quantiser (wq_pack.cu)
int pack_nf4(const float* W, int64_t N, int64_t K, uint8_t* packed, uint8_t* scales, cudaStream_t s);
int pack_nvfp4(const float* W, int64_t N, int64_t K, uint8_t* packed, uint8_t* scales, cudaStream_t s);
int pack_q4_0(const float* W, int64_t N, int64_t K, uint8_t* packed, uint8_t* scales, cudaStream_t s);
int pack_q8_0(const float* W, int64_t N, int64_t K, uint8_t* packed, uint8_t* scales, cudaStream_t s);
int pack_q4_1(const float* W, int64_t N, int64_t K, uint8_t* packed, uint8_t* scales, cudaStream_t s);
int pack_q5_0(const float* W, int64_t N, int64_t K, uint8_t* packed, uint8_t* scales, cudaStream_t s);
int pack_fp8(const float* W, int64_t N, int64_t K, uint8_t* packed, uint8_t* scales, cudaStream_t s);
int dequant(const uint8_t* packed, const uint8_t* scales, int fmt, int64_t N, int64_t K, float* out,
            cudaStream_t s);
int quant_act_nvfp4(const uint16_t* x, int64_t M, int64_t K, const float* g_in, uint8_t* codes,
                    uint8_t* scales, float* g_out, cudaStream_t s);
int take_status_pack();
int selftest_timeout(uint32_t polls, cudaStream_t s);  // bounded wait on a barrier nobody arrives on
int selftest_encoders(const float* in, int64_t n, uint8_t* out, cudaStream_t s);

// ---- linear: CUDA-core path (wq_simt.cu)
struct LinearArgs {
  const void* x;               // bf16 [M, K] (W4A16) -- unused for W4A4
  const uint8_t* act_codes;    // W4A4 activations
  const uint8_t* act_scales;
  const float* act_g;
  const uint8_t* packed;
  const uint8_t* scales;
  int fmt;
  int64_t M, N, K;
  const uint16_t* bias;
  void* y;                     // single output [M, N] (nout == 1, ld == N)
  bool out_f32;
  bool weights_static;         // may launch with programmatic dependent launch
  // Output destinations: columns [col_end[d-1], col_end[d]) of row m go to
  // ys[d] + m * ld[d] + (n - col_end[d-1]) (elements).  set_single_out() fills one destination.
  int nout;
  void* ys[WQ_OUT_MAX];
  int64_t ld[WQ_OUT_MAX];
  int64_t col_end[WQ_OUT_MAX];
};
inline void set_single_out(LinearArgs& a) {
  a.nout = 1;
  a.ys[0] = a.y;
  a.ld[0] = a.N;
  a.col_end[0] = a.N;
  for (int d = 1; d < WQ_OUT_MAX; ++d) { a.ys[d] = a.y; a.ld[d] = a.N; a.col_end[d] = a.N; }
}
// One Linear of any shape and output layout: the tensor-core paths where their rules hold,
// else the CUDA-core kernel.
int linear_one(const LinearArgs& a, cudaStream_t s);
int linear_simt(const LinearArgs& a, cudaStream_t s);
int take_status_simt();

// ---- linear: decode-sized single Linear on the CUDA cores (wq_gemv.cu)
constexpr int kGemvMaxM = 4;  // single Linears with up to this many activation rows take the GEMV
constexpr int kTcpDecodeMaxK = 2048;  // longer single decode Linears split K over a cluster instead
bool gemv_eligible(const LinearArgs& a);
int linear_gemv(const LinearArgs& a, cudaStream_t s);

// ---- linear: tensor-core paths (wq_tc.cu: decode split-K; wq_tcp.cu: persistent work list;
//      wq_w4a4.cu: block-scaled FP4)
constexpr int kGroupMax = WQ_GROUP_MAX;
bool tcp_eligible(const LinearArgs& a);
int linear_tcp(const LinearArgs* probs, int count, cudaStream_t s);
int take_status_tcp();
// return 1 = handled (status in *rc), 0 = shape not eligible for this path
int linear_tc(const LinearArgs& a, cudaStream_t s, int* rc);
int take_status_tc();
int linear_w4a4_tc(const LinearArgs& a, cudaStream_t s, int* rc);
int take_status_w4a4();
// NVFP4 W4A16 GEMM with 512-row activation tiles (wq_w4a16.cu); 0 = shape not taken
int linear_w4a16_tc(const LinearArgs& a, cudaStream_t s, int* rc);
int take_status_w4a16();

// driver entry point for tensor-map encoding (resolved once through the runtime)
bool encode_tmap_2d(void* tmap, CUtensorMapDataType dtype, const void* base, uint64_t inner, uint64_t outer,
                    uint64_t row_stride_bytes, uint32_t box_inner, uint32_t box_outer, CUtensorMapSwizzle swz);

}  // namespace wq
