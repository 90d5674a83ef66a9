// wq_tc.cu -- tensor-core fused dequantise-and-multiply for bf16 activations
// (NF4, NVFP4 W4A16, q4_0, q8_0), decode (M <= 16) and encoder-sized M alike.
//
// The operation (PR "asr: add a 4-bit nf4 option for the Whisper engine",
// "Why NF4 and not the NVFP4 snapshot"): y = x . dequant(W)^T + bias without
// ever writing the decoded W to memory -- unpacking to bf16 and calling an
// ordinary GEMM is what made the modelopt formats 4x slower there.
//
// Mapping onto sm_103a (transposed product, D^T = W_hat . x^T):
//   * MMA "A" = a 128-row tile of decoded weights.  Four dequant warps read the
//     packed codes that TMA staged in shared memory, decode them in registers
//     and store bf16 pairs straight into TENSOR MEMORY with tcgen05.st: the
//     decoded weights never touch shared memory.
//   * MMA "B" = BN rows of x, staged by TMA with the 128-byte swizzle the MMA
//     descriptor expects.
//   * tcgen05.mma.kind::f16 (bf16 x bf16 -> fp32) accumulates D[128 x BN] in
//     TMEM; one elected thread issues it.
//   * Decode (M <= 16, BN = 16) splits K over a thread-block cluster; the
//     partial D tiles are summed through distributed shared memory.
//   * Epilogue: tcgen05.ld, x global scale (NVFP4), + bias, bf16 (or fp32) store.
// All mbarrier waits are bounded (see wq_device.cuh).
#include <cuda.h>
#include <cuda_runtime.h>

#include <mutex>

#include "wq_device.cuh"
#include "wq_internal.h"
#include "wq_tc_common.cuh"

namespace wq {
namespace {

using namespace tc;
constexpr int kNA = 4;         // TMEM A-operand ring slots (32 columns each)
constexpr int kThreads = 192;  // warp 0 TMA, warp 1 MMA + TMEM owner, warps 2..5 dequant + epilogue

struct TcParams {
  const uint8_t* scales;
  const uint16_t* bias;
  void* y;
  int M, N, K;
  int out_f32;
  int ksplit;            // CTAs along K (a cluster when > 1)
  int weights_static;    // programmatic dependent launch: stream W before the dependency resolves
  ScalesLayout lay;
};

// Bounded wait that neither looks at the abort flag nor records a status: used after an abort, for
// the asynchronous copies and MMAs already issued to finish before the CTA releases its memory.
__device__ __forceinline__ void wait_quiet(uint64_t* bar, uint32_t parity) {
  for (uint32_t i = 0; i < kSpinLimit && !mbar_try_wait(bar, parity); ++i) {
  }
}

template <int BN, int STAGES, int FMT>
struct Smem {
  static constexpr int XB = BN * 128;                 // x stage bytes (BN rows x 64 bf16)
  static constexpr int WB = kRows * Fmt<FMT>::WB;     // packed weight stage bytes
  static constexpr int X_OFF = 0;
  static constexpr int W_OFF = X_OFF + STAGES * XB;
  static constexpr int LUT_OFF = W_OFF + STAGES * WB;  // 256 x float2
  static constexpr int BAR_OFF = LUT_OFF + 256 * 8;
  static constexpr int NBAR = 2 * STAGES + 2 * kNA + 2;
  static constexpr int MISC_OFF = BAR_OFF + NBAR * 8;  // tmem base, abort flag
  static constexpr int RED_OFF = (MISC_OFF + 16 + 15) / 16 * 16;
  static constexpr int RED_BYTES = (BN <= 16) ? kRows * (BN + 1) * 4 : 0;
  static constexpr int RB_OFF = RED_OFF + RED_BYTES;          // fp32 bias per tile row
  static constexpr int TOTAL = RB_OFF + kRows * 4 + 1024;     // + alignment slack
};

template <int BN>
struct TmemCols {
  static constexpr int D_COL = kNA * 32;  // D after the A ring
  static constexpr int USED = D_COL + BN;
  static constexpr int ALLOC = USED <= 256 ? 256 : 512;
};

template <int BN, int STAGES, int FMT>
__global__ void __launch_bounds__(kThreads, 1)
    wq_tc_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmW, TcParams p) {
  using S = Smem<BN, STAGES, FMT>;
  using T = TmemCols<BN>;
  constexpr uint32_t IDESC = idesc_bf16(kRows, BN);
  constexpr uint32_t STAGE_TX = (uint32_t)(S::XB + S::WB);

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + S::BAR_OFF);
  uint64_t* full = bars;
  uint64_t* empty = bars + STAGES;
  uint64_t* afull = bars + 2 * STAGES;
  uint64_t* aempty = afull + kNA;
  uint64_t* dfull = aempty + kNA;
  uint64_t* done = dfull + 1;  // every warp has finished
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + S::MISC_OFF);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + S::MISC_OFF + 4);
  float2* lut = reinterpret_cast<float2*>(smem + S::LUT_OFF);

  const int warp = (int)warp_id(), lane = (int)lane_id();
  const int n0 = blockIdx.x * kRows;
  const int m0 = blockIdx.y * BN;
  const int nchunk_total = p.K / kKS;
  const int z = blockIdx.z;
  const int kc_begin = (int)((int64_t)z * nchunk_total / p.ksplit);
  const int kc_end = (int)((int64_t)(z + 1) * nchunk_total / p.ksplit);
  const int nchunks = kc_end - kc_begin;

  if (threadIdx.x == 0) {
    for (int i = 0; i < STAGES; ++i) { mbar_init(&full[i], 1); mbar_init(&empty[i], 1 + 4); }
    for (int i = 0; i < kNA; ++i) { mbar_init(&afull[i], 4); mbar_init(&aempty[i], 1); }
    mbar_init(dfull, 1);
    mbar_init(done, kThreads / 32);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (FMT != WQ_Q8_0) {
    for (int i = threadIdx.x; i < 256; i += kThreads)
      lut[i] = make_float2(nibble_value<FMT>(i & 15u), nibble_value<FMT>(i >> 4));
  }
  if (warp == 1) tmem_alloc(tmem_slot, T::ALLOC);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  griddep_launch_dependents();

  if (warp == 0) {
    // ---------------- TMA producer
    if (lane == 0) {
      prefetch_tmap(&tmX);
      prefetch_tmap(&tmW);
      const int pre = p.weights_static ? (nchunks < STAGES ? nchunks : STAGES) : 0;
      for (int i = 0; i < pre; ++i) {  // weights first: they do not depend on the preceding kernel
        mbar_arrive_expect_tx(&full[i], STAGE_TX);
        tma_load_2d(smem + S::W_OFF + i * S::WB, &tmW, &full[i], (kc_begin + i) * Fmt<FMT>::WB, n0);
      }
      griddep_wait();
      for (int i = 0; i < pre; ++i)
        tma_load_2d(smem + S::X_OFF + i * S::XB, &tmX, &full[i], (kc_begin + i) * kKS, m0);
      int issued = pre;
      for (int i = pre; i < nchunks; ++i) {
        const int s = i % STAGES;
        if (i >= STAGES && !mbar_wait(&empty[s], ((i / STAGES) & 1) ^ 1, abort_flag)) break;
        mbar_arrive_expect_tx(&full[s], STAGE_TX);
        tma_load_2d(smem + S::W_OFF + s * S::WB, &tmW, &full[s], (kc_begin + i) * Fmt<FMT>::WB, n0);
        tma_load_2d(smem + S::X_OFF + s * S::XB, &tmX, &full[s], (kc_begin + i) * kKS, m0);
        issued = i + 1;
      }
      // stopped by a wait that ran out: let the copies of the stages in flight land before exit
      if (issued < nchunks)
        for (int c = issued - STAGES < 0 ? 0 : issued - STAGES; c < issued; ++c)
          wait_quiet(&full[c % STAGES], (c / STAGES) & 1);
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer
    if (lane == 0) {
      const uint32_t d_tmem = tmem_base + T::D_COL;
      for (int i = 0; i < nchunks; ++i) {
        const int s = i % STAGES, slot = i % kNA;
        if (!mbar_wait(&full[s], (i / STAGES) & 1, abort_flag)) break;
        if (!mbar_wait(&afull[slot], (i / kNA) & 1, abort_flag)) break;
        tc_fence_after();
        const uint32_t xaddr = smem_u32(smem + S::X_OFF + s * S::XB);
#pragma unroll
        for (int kk = 0; kk < kKS / 16; ++kk) {
          const uint64_t bdesc = smem_desc(xaddr + kk * 32, 16, 1024, 2);
          mma_bf16_ts(d_tmem, tmem_base + slot * 32 + kk * 8, bdesc, IDESC, (i | kk) != 0 ? 1u : 0u);
        }
        tc_commit(&aempty[slot]);
        tc_commit(&empty[s]);
      }
      tc_commit(dfull);
    }
  } else {
    // ---------------- dequant warps (then epilogue)
    const int q = warp & 3;           // TMEM lane quarter this warp may access
    const int r = q * 32 + lane;      // weight row within the tile
    const int64_t n = (int64_t)n0 + r;
    const bool row_ok = n < p.N;
    const uint32_t lane_base = (uint32_t)(q * 32) << 16;
    // Values that do not depend on the preceding kernel are requested before the first weight
    // tile lands, so their memory latency overlaps the weight stream's: the scale words of the
    // first kPre chunks of this row, the bias and the NVFP4 global scale.
    constexpr int kPre = 8;
    uint32_t sw[kPre];
#pragma unroll
    for (int i = 0; i < kPre; ++i)
      sw[i] = (i < nchunks && row_ok) ? scale_word<FMT>(p.scales, p.lay, p.K, n, kc_begin + i) : 0u;
    const float gsc = (FMT == WQ_NVFP4) ? *reinterpret_cast<const float*>(p.scales + p.lay.g_off) : 1.0f;
    const float bval = (p.bias && row_ok) ? bf16_bits_to_f32(p.bias[n]) : 0.0f;
    float* row_bias = reinterpret_cast<float*>(smem + S::RB_OFF);  // for the split-K reduction
    row_bias[r] = bval;
    for (int i = 0; i < nchunks; ++i) {
      const int s = i % STAGES, slot = i % kNA;
      uint32_t word = 0u;
#pragma unroll
      for (int j = 0; j < kPre; ++j)
        if (j == i) word = sw[j];
      if (i >= kPre && row_ok) word = scale_word<FMT>(p.scales, p.lay, p.K, n, kc_begin + i);
      if (!mbar_wait(&full[s], (i / STAGES) & 1, abort_flag)) break;
      if (i >= kNA && !mbar_wait(&aempty[slot], ((i / kNA) & 1) ^ 1, abort_flag)) break;
      constexpr int NW = Fmt<FMT>::WB / 16;  // 16-byte pieces of one row's 64 codes
      const uint4* src = reinterpret_cast<const uint4*>(smem + S::W_OFF + s * S::WB + r * Fmt<FMT>::WB);
      uint4 wv[NW];
#pragma unroll
      for (int k = 0; k < NW; ++k) wv[k] = src[k];
      uint32_t v[32];
      decode_span<FMT, 64, 1>(word, 0, wv, lut, 0, v);
      tmem_st32(tmem_base + lane_base + slot * 32, v);
      tc_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) { mbar_arrive(&afull[slot]); mbar_arrive(&empty[s]); }
    }

    // ---------------- epilogue
    const bool have_d = mbar_wait(dfull, 0, abort_flag);
    tc_fence_after();
    griddep_wait();
    float* red = reinterpret_cast<float*>(smem + S::RED_OFF);
    if (have_d) {
#pragma unroll 1
      for (int c0 = 0; c0 < BN; c0 += 16) {
        float acc[16];
        tmem_ld16(tmem_base + lane_base + T::D_COL + c0, acc);
        tc_wait_ld();
        if (p.ksplit == 1) {
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const int m = m0 + c0 + j;
            if (m < p.M && row_ok) {
              const float val = __fadd_rn(__fmul_rn(acc[j], gsc), bval);
              if (p.out_f32)
                reinterpret_cast<float*>(p.y)[(int64_t)m * p.N + n] = val;
              else
                reinterpret_cast<__nv_bfloat16*>(p.y)[(int64_t)m * p.N + n] = __float2bfloat16_rn(val);
            }
          }
        } else if (S::RED_BYTES) {
#pragma unroll
          for (int j = 0; j < 16; ++j) red[r * (BN + 1) + c0 + j] = acc[j];
        }
      }
    } else if (p.ksplit > 1 && S::RED_BYTES) {
      for (int j = 0; j < BN; ++j) red[r * (BN + 1) + j] = 0.0f;
    }
  }

  // ---------------- split-K: sum the cluster's partial tiles through DSMEM
  if (S::RED_BYTES && p.ksplit > 1) {
    __syncwarp();
    cluster_sync();
    if (warp >= 2) {
      const int ks = p.ksplit;
      const uint32_t rank = cluster_ctarank();
      const int r_lo = (int)(rank * kRows / ks), r_hi = (int)((rank + 1) * kRows / ks);
      const int rows = r_hi - r_lo;
      const int mcount = (p.M - m0) < BN ? (p.M - m0) : BN;
      const float gsc = (FMT == WQ_NVFP4) ? *reinterpret_cast<const float*>(p.scales + p.lay.g_off) : 1.0f;
      const float* row_bias = reinterpret_cast<const float*>(smem + S::RB_OFF);
      const uint32_t red_base = smem_u32(smem + S::RED_OFF);
      for (int idx = (int)threadIdx.x - 64; idx < rows * mcount; idx += 128) {
        const int j = idx / rows, rr = r_lo + idx % rows;
        const int64_t n = (int64_t)n0 + rr;
        if (n >= p.N) continue;
        const uint32_t off = red_base + (uint32_t)((rr * (BN + 1) + j) * 4);
        // every peer's partial is requested before the first is added, so the remote loads overlap
        // instead of paying the distributed-shared-memory latency once per peer
        float part[8];
#pragma unroll
        for (int pr = 0; pr < 8; ++pr)
          part[pr] = pr < ks ? ld_shared_cluster_f32(map_shared_rank(off, (uint32_t)pr)) : 0.0f;
        float sum = 0.0f;
#pragma unroll
        for (int pr = 0; pr < 8; ++pr) sum += part[pr];
        const float val = __fadd_rn(__fmul_rn(sum, gsc), row_bias[rr]);
        const int64_t m = m0 + j;
        if (p.out_f32)
          reinterpret_cast<float*>(p.y)[m * p.N + n] = val;
        else
          reinterpret_cast<__nv_bfloat16*>(p.y)[m * p.N + n] = __float2bfloat16_rn(val);
      }
    }
    __syncwarp();
    cluster_sync();
  }

  // Teardown: an mbarrier counts every warp; warp 1 then waits for the MMA issuer's commit after its
  // loop (all of its MMAs finished, also after an abort) and releases TMEM.  Bounded, and not cut
  // short by the abort flag: every other wait is bounded, so every warp arrives.
  tc_fence_before();
  __syncwarp();
  if (lane == 0) mbar_arrive(done);
  if (warp == 1) {
    wait_quiet(done, 0);
    if (*abort_flag) wait_quiet(dfull, 0);  // else the epilogue waited for it
    tc_fence_after();
    tmem_dealloc(tmem_base, T::ALLOC);
  }
}

template <int BN, int STAGES, int FMT>
int launch_tc(const LinearArgs& a, cudaStream_t s, int ksplit) {
  using S = Smem<BN, STAGES, FMT>;
  auto kern = wq_tc_kernel<BN, STAGES, FMT>;
  static std::once_flag once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(once, [&] {
    attr_err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, S::TOTAL);
    if (attr_err == cudaSuccess)
      attr_err = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
  });
  if (attr_err != cudaSuccess) return WQ_ERR_CUDA;

  alignas(64) CUtensorMap tmX, tmW;
  const uint64_t wrow = (uint64_t)(FMT == WQ_Q8_0 ? a.K : a.K / 2);
  if (!encode_tmap_2d(&tmX, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, a.x, (uint64_t)a.K, (uint64_t)a.M,
                      (uint64_t)a.K * 2, 64, BN, CU_TENSOR_MAP_SWIZZLE_128B))
    return WQ_ERR_CUDA;
  if (!encode_tmap_2d(&tmW, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.packed, wrow, (uint64_t)a.N, wrow,
                      Fmt<FMT>::WB, kRows, CU_TENSOR_MAP_SWIZZLE_NONE))
    return WQ_ERR_CUDA;

  TcParams p;
  p.scales = a.scales;
  p.bias = a.bias;
  p.y = a.y;
  p.M = (int)a.M;
  p.N = (int)a.N;
  p.K = (int)a.K;
  p.out_f32 = a.out_f32 ? 1 : 0;
  p.ksplit = ksplit;
  p.weights_static = a.weights_static ? 1 : 0;
  p.lay = scales_layout(FMT, a.N, a.K);

  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)((a.N + kRows - 1) / kRows), (unsigned)((a.M + BN - 1) / BN), (unsigned)ksplit);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = S::TOTAL;
  cfg.stream = s;
  cudaLaunchAttribute attrs[2];
  int na = 0;
  if (ksplit > 1) {
    attrs[na].id = cudaLaunchAttributeClusterDimension;
    attrs[na].val.clusterDim.x = 1;
    attrs[na].val.clusterDim.y = 1;
    attrs[na].val.clusterDim.z = (unsigned)ksplit;
    ++na;
  }
  if (a.weights_static) {
    attrs[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attrs[na].val.programmaticStreamSerializationAllowed = 1;
    ++na;
  }
  cfg.attrs = attrs;
  cfg.numAttrs = na;
  cudaError_t e = cudaLaunchKernelEx(&cfg, kern, tmX, tmW, p);
  count_launch();
  return e == cudaSuccess ? WQ_OK : WQ_ERR_CUDA;
}

constexpr int kDecodeStages = 12;

template <int FMT>
int dispatch_fmt(const LinearArgs& a, cudaStream_t s) {
  const int nchunks = (int)(a.K / kKS);
  const int ntiles = (int)((a.N + kRows - 1) / kRows);
  // split K over a cluster so that the grid covers the GPU (152 SMs)
  int ks = (2 * 152 + ntiles - 1) / ntiles;
  if (ks > 8) ks = 8;
  if (ks > nchunks) ks = nchunks;
  if (ks < 1) ks = 1;
  return launch_tc<16, kDecodeStages, FMT>(a, s, ks);
}

}  // namespace

int linear_tc(const LinearArgs& a, cudaStream_t s, int* rc) {
  // decode-sized M only; size rules of this path, anything else falls back to the CUDA-core kernel
  if (a.M > 16) return 0;
  if (a.K % kKS != 0 || a.K < kKS) return 0;
  if (a.M > 0x7FFFFFFF || a.N > 0x7FFFFFFF || a.K > 0x7FFFFFFF) return 0;
  if (((uintptr_t)a.x & 15u) != 0) return 0;
  switch (a.fmt) {
    case WQ_NF4: *rc = dispatch_fmt<WQ_NF4>(a, s); return 1;
    case WQ_NVFP4: *rc = dispatch_fmt<WQ_NVFP4>(a, s); return 1;
    case WQ_Q4_0: *rc = dispatch_fmt<WQ_Q4_0>(a, s); return 1;
    case WQ_Q8_0: *rc = dispatch_fmt<WQ_Q8_0>(a, s); return 1;
    default: return 0;
  }
}

int take_status_tc() {
  int v = 0, zero = 0;
  if (cudaMemcpyFromSymbol(&v, g_status, sizeof(int)) != cudaSuccess) return WQ_ERR_CUDA;
  cudaMemcpyToSymbol(g_status, &zero, sizeof(int));
  return v;
}

}  // namespace wq
