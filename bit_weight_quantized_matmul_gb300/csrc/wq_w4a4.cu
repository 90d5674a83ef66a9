// wq_w4a4.cu -- NVFP4 x NVFP4 (W4A4) GEMM on the block-scaled FP4 tensor cores.
//
// Model card "whisper-large-v3-turbo -- NVFP4", "What is quantized" and "Honest
// summary": E2M1 weights with an E4M3 scale per 16 values and an FP32 global scale,
// activations quantised the same way at runtime; on Blackwell the product runs as
// true W4A4.  Here:
//
//   y[m, n] = g_x * g_w * sum_k (e2m1(x) * s_x)[m, k] * (e2m1(w) * s_w)[n, k] + bias[n]
//
// Both operands stay packed: TMA stages the two codes per byte (128-byte swizzle) and
// tcgen05.mma.kind::mxf4nvf4.block_scale.scale_vec::4X multiplies them with their
// per-16 E4M3 block scales, which are held in tensor memory.  Nothing is decoded.
//
// Persistent CTA per SM over (weight tile, activation tile) items, warp-specialised:
//   warp 0      TMA: W codes [128 x 512], x codes [128 x 512], both tiles' scales
//   warp 1      TMEM owner, MMA issuer (8 MMAs of K = 64 per 512-element chunk)
//   warps 2..5  scale warps: chunk scales smem -> TMEM (replicated 32-lane layout)
//   warps 6..13 epilogue, two groups of four (columns 0..63 and 64..127 of D): tcgen05.ld,
//               * g_x * g_w, + bias, store y
// D is double-buffered in TMEM so an item's epilogue overlaps the next main loop.
// All waits are bounded.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <mutex>

#include "wq_device.cuh"
#include "wq_internal.h"
#include "wq_tc_common.cuh"

namespace wq {
namespace {

constexpr int kRows = 128;    // weight rows per tile (MMA M) == activation rows per tile (MMA N)
constexpr int kThreads = 448;
constexpr int kEpiGroups = 2;  // groups of four epilogue warps, each draining half of D's columns

// KC: K elements per chunk, 256 or 512 (one or two 128-byte swizzle rows of packed codes)
template <int KC>
struct Geo {
  static constexpr int kKC = KC;
  static constexpr int kSub = KC / 256;               // TMA boxes per operand per chunk
  static constexpr int kStages = KC == 512 ? 3 : 5;
  static constexpr int kCodeBytes = kRows * KC / 2;   // per operand per chunk
  static constexpr int kSFBytes = kRows * KC / 16;    // per operand per chunk
  static constexpr int kSFCols = 2 * 4 * (KC / 64);   // TMEM scale columns per chunk (both operands)
};

template <int N>
__device__ __forceinline__ void tmem_st_cols(uint32_t taddr, const uint32_t (&v)[N]);
template <>
__device__ __forceinline__ void tmem_st_cols<16>(uint32_t taddr, const uint32_t (&v)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(
          taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]), "r"(v[9]),
      "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15])
      : "memory");
}
template <>
__device__ __forceinline__ void tmem_st_cols<32>(uint32_t taddr, const uint32_t (&v)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]), "r"(v[9]),
      "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15]), "r"(v[16]), "r"(v[17]), "r"(v[18]),
      "r"(v[19]), "r"(v[20]), "r"(v[21]), "r"(v[22]), "r"(v[23]), "r"(v[24]), "r"(v[25]), "r"(v[26]), "r"(v[27]),
      "r"(v[28]), "r"(v[29]), "r"(v[30]), "r"(v[31])
      : "memory");
}

// Bounded wait that neither looks at the abort flag nor records a status: used after an abort, for
// the asynchronous copies and MMAs already issued to finish before the CTA releases its memory.
__device__ __forceinline__ void wait_quiet(uint64_t* bar, uint32_t parity) {
  for (uint32_t i = 0; i < kSpinLimit && !mbar_try_wait(bar, parity); ++i) {
  }
}

// One 16-column slab of the accumulator out to y through a 4 KB shared-memory buffer, for epilogue
// group G (128 threads, named barrier 1 + G): as tc::store_slab_bf16, with a barrier per group.
template <int G>
__device__ __forceinline__ void group_bar() {
  asm volatile("bar.sync %0, 128;" ::"n"(1 + G) : "memory");
}
template <int G>
__device__ __forceinline__ void store_slab_group(const float (&acc)[16], float gsc, float bval, int r,
                                                 uint16_t* stage, void* y, int64_t M, int64_t N, int64_t m0,
                                                 int64_t n0) {
  group_bar<G>();  // the group's previous slab has left the buffer
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    const float v = __fadd_rn(__fmul_rn(acc[j], gsc), bval);
    stage[j * 128 + r] = __bfloat16_as_ushort(__float2bfloat16_rn(v));
  }
  group_bar<G>();
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

struct W4Params {
  const uint8_t* w_scales;   // weight scales blob (E4M3 [N, K/16] | pad | g)
  const float* g_x;          // activation global scale (device)
  const uint16_t* bias;
  void* y;
  int M, N, K;
  int ntiles, mtiles, total_items, out_f32;
  int weights_static;  // programmatic dependent launch: weight tiles stream before the dependency resolves
  uint32_t g_off;
};

struct W4Maps {
  CUtensorMap wc, xc, ws, xs;  // codes and scale maps of W and x
};

template <int KC>
struct Lay {
  static constexpr int kStages = Geo<KC>::kStages, kCodeBytes = Geo<KC>::kCodeBytes, kSFBytes = Geo<KC>::kSFBytes;
  static constexpr int A_OFF = 0;                              // W codes  [stage]
  static constexpr int B_OFF = A_OFF + kStages * kCodeBytes;   // x codes  [stage]
  static constexpr int SA_OFF = B_OFF + kStages * kCodeBytes;  // W scales [stage]
  static constexpr int SB_OFF = SA_OFF + kStages * kSFBytes;   // x scales [stage]
  static constexpr int BAR_OFF = SB_OFF + kStages * kSFBytes;
  static constexpr int NBAR = 3 * kStages + 6;
  static constexpr int MISC_OFF = BAR_OFF + NBAR * 8;
  static constexpr int Y_OFF = (MISC_OFF + 16 + 127) / 128 * 128;  // 4 KB output slab per epilogue group
  static constexpr int TOTAL = Y_OFF + 2 * 16 * kRows * 2 + 1024;
  static_assert(TOTAL <= 227 * 1024, "shared memory budget");
};

// TMEM columns: D double buffer [0, 256), then one scale slot per shared-memory stage: per chunk
// KC / 64 MMAs x (4 columns of weight scales + 4 of activation scales)
constexpr int kDCol = 0;
constexpr int kSFCol = 2 * kRows;
constexpr int kTmemCols = 512;
static_assert(kSFCol + Geo<512>::kStages * Geo<512>::kSFCols <= kTmemCols, "TMEM budget");
static_assert(kSFCol + Geo<256>::kStages * Geo<256>::kSFCols <= kTmemCols, "TMEM budget");

template <int KC>
__global__ void __launch_bounds__(kThreads, 1)
    wq_w4a4_kernel(const __grid_constant__ W4Maps maps, const __grid_constant__ W4Params p) {
  using Lay = wq::Lay<KC>;
  constexpr int kKC = KC, kSub = Geo<KC>::kSub, kStages = Geo<KC>::kStages;
  constexpr int kCodeBytes = Geo<KC>::kCodeBytes, kSFBytes = Geo<KC>::kSFBytes, kSFCols = Geo<KC>::kSFCols;
  constexpr uint32_t IDESC = idesc_nvf4(kRows, kRows);
  constexpr uint32_t STAGE_TX = 2 * kCodeBytes + 2 * kSFBytes;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Lay::BAR_OFF);
  uint64_t* full = bars;
  uint64_t* empty = bars + kStages;
  uint64_t* sffull = bars + 2 * kStages;  // stage s's scales are in TMEM slot s
  uint64_t* dfull = sffull + kStages;      // [2]
  uint64_t* dempty = dfull + 2;          // [2]
  uint64_t* done = dempty + 2;           // every warp has finished
  uint64_t* drain = done + 1;            // the MMA issuer's last commit: all of its MMAs finished
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + Lay::MISC_OFF);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + Lay::MISC_OFF + 4);
  const int warp = (int)warp_id(), lane = (int)lane_id();

  if (threadIdx.x == 0) {
    for (int i = 0; i < kStages; ++i) { mbar_init(&full[i], 1); mbar_init(&empty[i], 1 + 4); }
    mbar_init(done, kThreads / 32);
    mbar_init(drain, 1);
    for (int i = 0; i < kStages; ++i) mbar_init(&sffull[i], 4);
    for (int i = 0; i < 2; ++i) { mbar_init(&dfull[i], 1); mbar_init(&dempty[i], 4 * kEpiGroups); }
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) tmem_alloc(tmem_slot, kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  griddep_launch_dependents();

  // a last chunk that runs past K reads TMA's zero fill: zero codes with zero scales add nothing
  const int nch = (p.K + kKC - 1) / kKC;
  const int total = p.total_items;
  if (warp == 0) {
    // ---------------------------------------------- TMA producer
    if (lane == 0) {
      prefetch_tmap(&maps.wc);
      prefetch_tmap(&maps.xc);
      prefetch_tmap(&maps.ws);
      prefetch_tmap(&maps.xs);
      // weight tiles (codes + block scales) of the first stages do not depend on the preceding
      // kernel when the caller promised static weights: they stream while it finishes (e.g. while
      // the activation quantiser runs); the activation tiles wait for it
      auto load_w = [&](int s, int c, int nt) {
#pragma unroll
        for (int b = 0; b < kSub; ++b)  // [128 rows x 128 B] boxes, 128-byte swizzle
          tma_load_2d(smem + Lay::A_OFF + s * kCodeBytes + b * 16384, &maps.wc, &full[s], c * (kKC / 2) + b * 128,
                      nt * kRows);
        tma_load_2d(smem + Lay::SA_OFF + s * kSFBytes, &maps.ws, &full[s], c * (kKC / 16), nt * kRows);
      };
      auto load_x = [&](int s, int c, int mt) {
#pragma unroll
        for (int b = 0; b < kSub; ++b)
          tma_load_2d(smem + Lay::B_OFF + s * kCodeBytes + b * 16384, &maps.xc, &full[s], c * (kKC / 2) + b * 128,
                      mt * kRows);
        tma_load_2d(smem + Lay::SB_OFF + s * kSFBytes, &maps.xs, &full[s], c * (kKC / 16), mt * kRows);
      };
      int pre = 0;
      if (p.weights_static) {
        for (int it = blockIdx.x; it < total && pre < kStages; it += gridDim.x)
          for (int c = 0; c < nch && pre < kStages; ++c, ++pre) {
            mbar_arrive_expect_tx(&full[pre], STAGE_TX);
            load_w(pre, c, it % p.ntiles);
          }
      }
      griddep_wait();
      int g = 0;
      bool ok = true;
      for (int it = blockIdx.x; it < total && ok; it += gridDim.x) {
        const int nt = it % p.ntiles, mt = it / p.ntiles;
        for (int c = 0; c < nch; ++c, ++g) {
          const int s = g % kStages;
          if (g >= pre) {
            if (g >= kStages && !mbar_wait(&empty[s], ((g / kStages) & 1) ^ 1, abort_flag)) { ok = false; break; }
            mbar_arrive_expect_tx(&full[s], STAGE_TX);
            load_w(s, c, nt);
          }
          load_x(s, c, mt);
        }
      }
      // stopped by a wait that ran out: let the copies of the stages in flight land before exit
      if (!ok)
        for (int c = g - kStages < 0 ? 0 : g - kStages; c < g; ++c) wait_quiet(&full[c % kStages], (c / kStages) & 1);
    }
  } else if (warp == 1) {
    // ---------------------------------------------- MMA issuer
    if (lane == 0) {
      const uint64_t a_desc0 = smem_desc(smem_u32(smem + Lay::A_OFF), 16, 1024, 2);
      const uint64_t b_desc0 = smem_desc(smem_u32(smem + Lay::B_OFF), 16, 1024, 2);
      int g = 0, n_it = 0;
      bool ok = true;
      for (int it = blockIdx.x; it < total && ok; it += gridDim.x, ++n_it) {
        const int buf = n_it & 1;
        if (n_it >= 2 && !mbar_wait(&dempty[buf], ((n_it >> 1) & 1) ^ 1, abort_flag)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + kDCol + buf * kRows;
        for (int c = 0; c < nch; ++c, ++g) {
          const int s = g % kStages;
          // the scale warps waited for stage s's TMA transaction before they filled its scale slot
          if (!mbar_wait(&sffull[s], (g / kStages) & 1, abort_flag)) { ok = false; break; }
          tc_fence_after();
          // descriptors differ from stage 0's only in the start-address field (16-byte units)
          const uint64_t ad = a_desc0 + (uint64_t)((s * kCodeBytes) >> 4);
          const uint64_t bd = b_desc0 + (uint64_t)((s * kCodeBytes) >> 4);
          const uint32_t sfa = tmem_base + kSFCol + s * kSFCols;
#pragma unroll
          for (int i = 0; i < kKC / 64; ++i) {  // K = 64 E2M1 values (32 bytes) per MMA
            constexpr uint32_t kOff16[8] = {0, 2, 4, 6, 1024, 1026, 1028, 1030};  // (i/4)*16384 + (i%4)*32, /16
            mma_nvf4_ss(d_tmem, ad + kOff16[i], bd + kOff16[i], IDESC, sfa + i * 4, sfa + kSFCols / 2 + i * 4,
                        (c | i) != 0 ? 1u : 0u);
          }
          // one commit frees both the shared-memory stage (with the scale warps' arrivals) and,
          // through the producer's wait before it refills the stage, the TMEM scale slot
          tc_commit(&empty[s]);
        }
        if (ok) tc_commit(&dfull[buf]);
      }
      // after an abort: a commit that tracks every MMA this thread issued, for the teardown's wait
      if (!ok || *abort_flag) tc_commit(drain);
    }
  } else if (warp < 6) {
    // ---------------------------------------------- scale warps: smem [128 rows x KC/16 B] -> TMEM
    // For MMA i of a chunk, lane r of every 32-lane quarter holds, in column 4 i + j (j = 0..3),
    // the four E4M3 scales (K blocks 4i .. 4i+3) of row 32 j + r -- the replicated layout that a
    // 32x128b.warpx4 copy of a 512-byte scale atom produces.  Each thread reads its four rows'
    // scale bytes as 16-byte vectors and writes a whole chunk's columns with one store per operand.
    const int q = warp & 3;
    const uint32_t lane_base = (uint32_t)(q * 32) << 16;
    constexpr int NW = kKC / 64;  // 32-bit scale words per row per chunk (one per MMA)
    int g = 0;
    bool ok = true;
    for (int it = blockIdx.x; it < total && ok; it += gridDim.x) {
      for (int c = 0; c < nch; ++c, ++g) {
        // stage s's TMA transaction completing implies that the producer saw the MMAs of chunk
        // g - kStages finish (it waited for them before refilling the stage): scale slot s is free
        const int s = g % kStages, slot = s;
        if (!mbar_wait(&full[s], (g / kStages) & 1, abort_flag)) { ok = false; break; }
#pragma unroll
        for (int op = 0; op < 2; ++op) {
          const uint8_t* sbase = smem + (op == 0 ? Lay::SA_OFF : Lay::SB_OFF) + s * kSFBytes;
          uint32_t v[4 * NW];
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const uint4* row = reinterpret_cast<const uint4*>(sbase + (32 * j + lane) * (kKC / 16));
#pragma unroll
            for (int h = 0; h < NW / 4; ++h) {
              const uint4 w = row[h];
              v[(4 * h + 0) * 4 + j] = w.x;
              v[(4 * h + 1) * 4 + j] = w.y;
              v[(4 * h + 2) * 4 + j] = w.z;
              v[(4 * h + 3) * 4 + j] = w.w;
            }
          }
          tmem_st_cols<4 * NW>(tmem_base + lane_base + kSFCol + slot * kSFCols + op * (kSFCols / 2), v);
        }
        tc_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) { mbar_arrive(&sffull[slot]); mbar_arrive(&empty[s]); }
      }
    }
  } else {
    // ---------------------------------------------- epilogue
    const int q = warp & 3;
    const int r = q * 32 + lane;
    const uint32_t lane_base = (uint32_t)(q * 32) << 16;
    const int grp = (warp - 6) / 4;  // this group's columns: [64 grp, 64 grp + 64)
    griddep_wait();
    const float gw = *reinterpret_cast<const float*>(p.w_scales + p.g_off);
    const float gs = __fmul_rn(*p.g_x, gw);
    int n_it = 0;
    for (int it = blockIdx.x; it < total; it += gridDim.x, ++n_it) {
      const int nt = it % p.ntiles, mt = it / p.ntiles;
      const int buf = n_it & 1;
      const int64_t n = (int64_t)nt * kRows + r;
      const bool row_ok = n < p.N;
      const float bval = (p.bias && row_ok) ? bf16_bits_to_f32(p.bias[n]) : 0.0f;
      if (!mbar_wait(&dfull[buf], (n_it >> 1) & 1, abort_flag)) break;
      tc_fence_after();
      const int m0 = mt * kRows;
      uint16_t* ystage = reinterpret_cast<uint16_t*>(smem + Lay::Y_OFF) + grp * 16 * kRows;
      // 32 columns per tensor-memory wait; each 16-column slab goes out through this group's 4 KB
      // buffer, guarded by the group's own named barrier (ids 1 and 2)
#pragma unroll 1
      for (int c1 = grp * (kRows / kEpiGroups); c1 < (grp + 1) * (kRows / kEpiGroups); c1 += 32) {
        float acc[2][16];
        tmem_ld16(tmem_base + lane_base + kDCol + buf * kRows + c1, acc[0]);
        tmem_ld16(tmem_base + lane_base + kDCol + buf * kRows + c1 + 16, acc[1]);
        tc_wait_ld();
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int c0 = c1 + 16 * h;
          if (!p.out_f32) {
            if (grp == 0)
              store_slab_group<0>(acc[h], gs, bval, r, ystage, p.y, p.M, p.N, m0 + c0, (int64_t)nt * kRows);
            else
              store_slab_group<1>(acc[h], gs, bval, r, ystage, p.y, p.M, p.N, m0 + c0, (int64_t)nt * kRows);
          } else if (row_ok) {
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              const int m = m0 + c0 + j;
              if (m < p.M)
                reinterpret_cast<float*>(p.y)[(int64_t)m * p.N + n] = __fadd_rn(__fmul_rn(acc[h][j], gs), bval);
            }
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&dempty[buf]);
    }
  }

  // Teardown: an mbarrier counts every warp (a CTA-wide bar.sync after lane-divergent roles is not
  // relied on), then warp 1 waits for the MMA issuer's last commit and releases TMEM.  The waits
  // are bounded and not cut short by the abort flag: every other wait is bounded, so every warp
  // arrives.
  tc_fence_before();
  __syncwarp();
  if (lane == 0) mbar_arrive(done);
  if (warp == 1) {
    wait_quiet(done, 0);
    if (*abort_flag) wait_quiet(drain, 0);  // else the epilogue saw every MMA finish
    tc_fence_after();
    tmem_dealloc(tmem_base, kTmemCols);
  }
}

int num_sms_w4() {
  static int n = 0;
  static std::once_flag once;
  std::call_once(once, [] {
    int dev = 0;
    cudaGetDevice(&dev);
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) n = 148;
  });
  return n;
}

template <int KC>
int launch_w4a4(const LinearArgs& a, cudaStream_t s, int* rc) {
  using Lay = wq::Lay<KC>;
  auto kern = wq_w4a4_kernel<KC>;
  static std::once_flag once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(once, [&] {
    attr_err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Lay::TOTAL);
  });
  if (attr_err != cudaSuccess) { *rc = WQ_ERR_CUDA; return 1; }
  alignas(64) W4Maps maps;
  const uint64_t kb = (uint64_t)a.K / 2, ks = (uint64_t)a.K / 16;
  bool ok = encode_tmap_2d(&maps.wc, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.packed, kb, (uint64_t)a.N, kb, 128, kRows,
                           CU_TENSOR_MAP_SWIZZLE_128B) &&
            encode_tmap_2d(&maps.xc, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.act_codes, kb, (uint64_t)a.M, kb, 128,
                           kRows, CU_TENSOR_MAP_SWIZZLE_128B) &&
            encode_tmap_2d(&maps.ws, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.scales, ks, (uint64_t)a.N, ks, KC / 16, kRows,
                           CU_TENSOR_MAP_SWIZZLE_NONE) &&
            encode_tmap_2d(&maps.xs, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.act_scales, ks, (uint64_t)a.M, ks, KC / 16,
                           kRows, CU_TENSOR_MAP_SWIZZLE_NONE);
  if (!ok) { *rc = WQ_ERR_CUDA; return 1; }
  W4Params p;
  p.w_scales = a.scales;
  p.g_x = a.act_g;
  p.bias = a.bias;
  p.y = a.y;
  p.M = (int)a.M;
  p.N = (int)a.N;
  p.K = (int)a.K;
  p.ntiles = (int)((a.N + kRows - 1) / kRows);
  p.mtiles = (int)((a.M + kRows - 1) / kRows);
  p.total_items = p.ntiles * p.mtiles;
  p.out_f32 = a.out_f32 ? 1 : 0;
  p.weights_static = a.weights_static ? 1 : 0;
  p.g_off = (uint32_t)scales_layout(WQ_NVFP4, a.N, a.K).g_off;

  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)std::min(p.total_items, num_sms_w4()), 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = Lay::TOTAL;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  cfg.numAttrs = 0;
  if (a.weights_static) {
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
  }
  cudaError_t e = cudaLaunchKernelEx(&cfg, kern, maps, p);
  count_launch();
  *rc = e == cudaSuccess ? WQ_OK : WQ_ERR_CUDA;
  return 1;
}

}  // namespace

int linear_w4a4_tc(const LinearArgs& a, cudaStream_t s, int* rc) {
  // size rules: scale rows of a multiple of 16 bytes (K % 256 == 0); decode-sized M stays on the CUDA cores
  if (a.M <= 16 || a.K % 256 != 0 || a.M > 0x7FFFFFFF || a.N > 0x7FFFFFFF || a.K > 0x7FFFFFFF) return 0;
  // 512-element chunks when they tile K exactly, else 256
  return a.K % 512 == 0 ? launch_w4a4<512>(a, s, rc) : launch_w4a4<256>(a, s, rc);
}

int take_status_w4a4() {
  int v = 0, zero = 0;
  if (cudaMemcpyFromSymbol(&v, g_status, sizeof(int)) != cudaSuccess) return WQ_ERR_CUDA;
  cudaMemcpyToSymbol(g_status, &zero, sizeof(int));
  return v;
}

}  // namespace wq
