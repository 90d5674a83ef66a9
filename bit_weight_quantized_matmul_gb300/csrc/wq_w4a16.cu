// wq_w4a16.cu -- NVFP4 weights x bf16 activations (W4A16) GEMM for encoder-sized M: each weight
// tile is dequantised once into shared memory, and the accumulator is double-buffered in TMEM.
//
// Model card "whisper-large-v3-turbo -- NVFP4", "What is quantized": E2M1 weights with an E4M3
// scale per 16 values and an FP32 global scale g; with 16-bit activations the product is
//
//   y[m, n] = g * sum_k x[m, k] * (e2m1(w) * s_w)[n, k] + bias[n]
//
// e2m1 * e4m3 has at most 5 significant bits, so each weight is exact in bf16; the MMA runs
// tcgen05.mma.kind::f16 (bf16 x bf16, fp32 accumulate) and g is applied in the epilogue.
//
// A tile of 128 weight rows is decoded into shared memory (the canonical 128-byte-swizzled K-major
// layout the MMA reads) rather than into TMEM, so TMEM holds only accumulators: two of BM columns,
// and a tile's epilogue overlaps the next tile's main loop.  Per K step one N = BM MMA over a BM-row
// activation tile: BM = 256, or 128 where 256-row tiles would leave SMs idle (each weight tile is then
// decoded once per 128 rows instead of 256).  (Two N = 256 MMAs over a 512-row tile with one
// 512-column accumulator measured slower: no overlap of the epilogue and fewer, larger items.)
// Persistent CTA per SM over (weight tile, activation tile) items, warp-specialised:
//   warp 0       TMA: activation tiles [BM x 64] (a stage is released by the MMAs reading it)
//   warp 1       TMEM owner, MMA issuer (4 K steps per 64-element chunk)
//   warps 2..17  dequant, four groups of four each taking every fourth chunk (four chunks decode at
//                once, each group in its own A slot): E2M1 -> bf16 x E4M3 block scale, a whole
//                64-element row chunk per thread, written swizzled into the shared-memory A ring
//   warps 18..21 epilogue: tcgen05.ld, * g, + bias, bf16 y through a 4 KB staging slab
//   warp 22      TMA: weight codes [128 x 32 B] on a ring of their own, released by the dequant
//                warps, so the decode runs ahead of the MMAs by up to the A ring's depth
// All waits are bounded; after a wait runs out the roles stop and the issued copies and MMAs are
// drained before TMEM is released.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <mutex>

#include "wq_device.cuh"
#include "wq_internal.h"
#include "wq_tc_common.cuh"

namespace wq {
namespace {

constexpr int kRows = 128;       // weight rows per tile (MMA M)
constexpr int kKC = 64;          // K elements per chunk: one 128-byte row of bf16
constexpr int kNA = 4;           // decoded weight (A) slots (fills shared memory: 222 KB)
constexpr int kDeqWarps = 16;                  // four groups of four, every fourth chunk
constexpr int kDeqGroups = 4;
constexpr int kGroupWarps = kDeqWarps / kDeqGroups;
constexpr int kParts = kGroupWarps / 4;        // parts of a 64-element chunk
constexpr int kEPT = kKC / kParts;             // elements a dequant thread decodes per chunk
constexpr int kEpiGroups = 1;                  // groups of four epilogue warps
constexpr int kEpiWarp0 = 2 + kDeqWarps;
constexpr int kWProdWarp = kEpiWarp0 + 4 * kEpiGroups;  // weight-code TMA
constexpr int kThreads = (kWProdWarp + 1) * 32;
static_assert(kEPT == 16 || kEPT == 32 || kEPT == 64, "dequant part");

__device__ __forceinline__ void mma_bf16_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                            uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}"
      ::"r"(d_tmem), "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Bounded wait that neither looks at the abort flag nor records a status: used after an abort, for
// the asynchronous copies and MMAs already issued to finish before the CTA releases its memory.
__device__ __forceinline__ void wait_quiet(uint64_t* bar, uint32_t parity) {
  for (uint32_t i = 0; i < kSpinLimit && !mbar_try_wait(bar, parity); ++i) {
  }
}

template <int G>
__device__ __forceinline__ void group_bar() {
  asm volatile("bar.sync %0, 128;" ::"n"(1 + G) : "memory");
}

// One 16-column slab of an accumulator half (TMEM lanes = 128 weight rows n0.., columns = 16
// activation rows m0..) to y through this group's 4 KB buffer: each thread scales and writes its 16
// values into stage[m][r], then the threads copy the [16 x 128] bf16 slab out as 256-byte rows.
template <int G>
__device__ __forceinline__ void store_slab(const float (&acc)[16], float g, float bval, int r, uint16_t* stage,
                                           void* y, int64_t M, int64_t N, int64_t m0, int64_t n0) {
  group_bar<G>();  // the group's previous slab has left the buffer
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    const float v = __fadd_rn(__fmul_rn(acc[j], g), bval);
    stage[j * 128 + r] = __bfloat16_as_ushort(__float2bfloat16_rn(v));
  }
  group_bar<G>();
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

struct W16Params {
  const uint8_t* scales;   // weight scales blob (E4M3 [N, K/16] | pad | g)
  const uint16_t* bias;
  void* y;
  int M, N, K;
  int ntiles, mtiles, total_items, out_f32;
  int weights_static;
  uint32_t g_off;
};

struct W16Maps {
  CUtensorMap x, w;
};

// BM: activation rows per tile (the MMA's N); two BM-column accumulators in TMEM
template <int BM>
struct Lay16 {
  static_assert(BM == 256 || BM == 128, "activation tile");
  static constexpr int NDB = 2;
  static constexpr int TMEM_COLS = NDB * BM;
  static constexpr int STAGES = BM == 256 ? 4 : 6;   // activation stages
  static constexpr int WSTAGES = BM == 256 ? 4 : 8;  // weight-code stages
  static constexpr int XB = BM * 128;                // activation stage bytes
  static constexpr int WB = kRows * (kKC / 2);     // weight-code stage bytes
  static constexpr int AB = kRows * 128;           // decoded weight slot bytes
  static constexpr int X_OFF = 0;
  static constexpr int A_OFF = X_OFF + STAGES * XB;
  static constexpr int W_OFF = A_OFF + kNA * AB;
  static constexpr int Y_OFF = W_OFF + WSTAGES * WB;
  static constexpr int BAR_OFF = Y_OFF + 2 * 16 * kRows * 2;
  static constexpr int NBAR = 2 * STAGES + 2 * WSTAGES + 2 * kNA + 6;
  static constexpr int MISC_OFF = BAR_OFF + NBAR * 8;
  static constexpr int TOTAL = MISC_OFF + 16 + 1024;
  static_assert(TOTAL <= 227 * 1024, "shared memory budget");
};

template <int BM>
__global__ void __launch_bounds__(kThreads, 1)
    wq_w4a16_kernel(const __grid_constant__ W16Maps maps, const __grid_constant__ W16Params p) {
  using L = Lay16<BM>;
  constexpr uint32_t IDESC = idesc_bf16(kRows, BM);
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::BAR_OFF);
  uint64_t* full = bars;                      // [L::STAGES] activation tile landed
  uint64_t* empty = bars + L::STAGES;         // [L::STAGES] the MMAs reading it finished
  uint64_t* wfull = bars + 2 * L::STAGES;     // [L::WSTAGES] weight codes landed
  uint64_t* wempty = wfull + L::WSTAGES;      // [L::WSTAGES] weight codes decoded
  uint64_t* afull = wempty + L::WSTAGES;      // [kNA] decoded weights written
  uint64_t* aempty = afull + kNA;         // [kNA] the MMAs reading them finished
  uint64_t* dfull = aempty + kNA;         // [2] accumulator complete
  uint64_t* dempty = dfull + 2;           // [2] accumulator read out
  uint64_t* done = dempty + 2;            // every warp has finished
  uint64_t* drain = done + 1;             // the MMA issuer's last commit
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::MISC_OFF);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::MISC_OFF + 4);
  const int warp = (int)warp_id(), lane = (int)lane_id();

  if (threadIdx.x == 0) {
    for (int i = 0; i < L::STAGES; ++i) { mbar_init(&full[i], 1); mbar_init(&empty[i], 1); }
    for (int i = 0; i < L::WSTAGES; ++i) { mbar_init(&wfull[i], 1); mbar_init(&wempty[i], kGroupWarps); }
    for (int i = 0; i < kNA; ++i) { mbar_init(&afull[i], kGroupWarps); mbar_init(&aempty[i], 1); }
    for (int i = 0; i < 2; ++i) { mbar_init(&dfull[i], 1); mbar_init(&dempty[i], 4 * kEpiGroups); }
    mbar_init(done, kThreads / 32);
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) tmem_alloc(tmem_slot, L::TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  griddep_launch_dependents();

  const int nch = p.K / kKC;
  const int total = p.total_items;
  if (warp == 0) {
    // ---------------------------------------------- TMA producer: activations
    if (lane == 0) {
      prefetch_tmap(&maps.x);
      griddep_wait();
      int g = 0;
      bool ok = true;
      for (int it = blockIdx.x; it < total && ok; it += gridDim.x) {
        const int mt = it / p.ntiles;
        for (int c = 0; c < nch; ++c, ++g) {
          const int s = g % L::STAGES;
          if (g >= L::STAGES && !mbar_wait(&empty[s], ((g / L::STAGES) & 1) ^ 1, abort_flag)) { ok = false; break; }
          mbar_arrive_expect_tx(&full[s], L::XB);
          tma_load_2d(smem + L::X_OFF + s * L::XB, &maps.x, &full[s], c * kKC, mt * BM);
        }
      }
      // stopped by a wait that ran out: let the copies of the stages in flight land before exit
      if (!ok)
        for (int c = g - L::STAGES < 0 ? 0 : g - L::STAGES; c < g; ++c) wait_quiet(&full[c % L::STAGES], (c / L::STAGES) & 1);
    }
  } else if (warp == 1) {
    // ---------------------------------------------- MMA issuer
    if (lane == 0) {
      const uint64_t a_desc0 = smem_desc(smem_u32(smem + L::A_OFF), 16, 1024, 2);
      const uint64_t x_desc0 = smem_desc(smem_u32(smem + L::X_OFF), 16, 1024, 2);
      int g = 0, n_it = 0;
      bool ok = true;
      for (int it = blockIdx.x; it < total && ok; it += gridDim.x, ++n_it) {
        const int buf = n_it % L::NDB;
        if (n_it >= L::NDB && !mbar_wait(&dempty[buf], ((n_it / L::NDB) & 1) ^ 1, abort_flag)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + buf * BM;
        for (int c = 0; c < nch; ++c, ++g) {
          const int s = g % L::STAGES, slot = g % kNA;
          if (!mbar_wait(&afull[slot], (g / kNA) & 1, abort_flag)) { ok = false; break; }
          if (!mbar_wait(&full[s], (g / L::STAGES) & 1, abort_flag)) { ok = false; break; }
          tc_fence_after();
          const uint64_t ad = a_desc0 + (uint64_t)((slot * L::AB) >> 4);
          const uint64_t xd = x_desc0 + (uint64_t)((s * L::XB) >> 4);
#pragma unroll
          for (int kk = 0; kk < kKC / 16; ++kk)  // K = 16 bf16 (32 bytes) per MMA
            mma_bf16_ss(d_tmem, ad + kk * 2, xd + kk * 2, IDESC, (c | kk) != 0 ? 1u : 0u);
          tc_commit(&aempty[slot]);
          tc_commit(&empty[s]);
        }
        if (ok) tc_commit(&dfull[buf]);
      }
      // after an abort: a commit that tracks every MMA this thread issued, for the teardown's wait
      if (!ok || *abort_flag) tc_commit(drain);
    }
  } else if (warp < kEpiWarp0) {
    // ---------------------------------------------- dequant warps
    // Group dg = (w - 2) / 4 decodes the chunks g with g % 4 == dg (the stage and slot indices follow
    // g modulo multiples of 4, so each group has its own share of both rings); within it, warp w
    // decodes rows 32 q + lane (q = (w - 2) % 4): kEPT / 2 code bytes and kEPT / 16 E4M3 scales per
    // row and chunk, kEPT bf16 values of the row's 64.
    static_assert(kNA % kDeqGroups == 0 && L::WSTAGES % kDeqGroups == 0, "rings split between the groups");
    const int dw = warp - 2;
    const int dg = dw / kGroupWarps, q = dw & 3, pt = (dw % kGroupWarps) >> 2;
    const int r = q * 32 + lane;
    const int nb16 = p.K / 16;
    constexpr int SPC = kEPT / 16;  // scale bytes per part
    int gb = 0;  // running chunk index of the item's first chunk
    bool ok = true;
    for (int it = blockIdx.x; it < total && ok; it += gridDim.x, gb += nch) {
      const int nt = it % p.ntiles;
      const int64_t n = (int64_t)nt * kRows + r;
      const bool row_ok = n < p.N;
      const uint8_t* srow = p.scales + (row_ok ? n : 0) * nb16 + pt * SPC;
      auto scale_bytes = [&](int c) -> uint32_t {  // this part's scales of chunk c
        if (!row_ok) return 0u;
        return SPC == 4   ? __ldg(reinterpret_cast<const uint32_t*>(srow + 4 * c))
               : SPC == 2 ? (uint32_t)__ldg(reinterpret_cast<const uint16_t*>(srow + 4 * c))
                          : (uint32_t)__ldg(srow + 4 * c);
      };
      const int c0 = (dg - gb % kDeqGroups + kDeqGroups) % kDeqGroups;  // this group's first chunk of the item
      uint32_t sc_next = c0 < nch ? scale_bytes(c0) : 0u;
      for (int c = c0; c < nch; c += kDeqGroups) {
        const int g = gb + c;
        const int ws = g % L::WSTAGES, slot = g % kNA;
        const uint32_t sc = sc_next;
        if (c + kDeqGroups < nch) sc_next = scale_bytes(c + kDeqGroups);
        if (!mbar_wait(&wfull[ws], (g / L::WSTAGES) & 1, abort_flag)) { ok = false; break; }
        if (g >= kNA && !mbar_wait(&aempty[slot], ((g / kNA) & 1) ^ 1, abort_flag)) { ok = false; break; }
        // this part's code bytes: 16-byte piece (kEPT / 2 bytes) pt * kEPT / 32 of the 32-byte row,
        // stored with TMA's 32-byte swizzle (address bit 4 ^= bit 7)
        const int boff = pt * (kEPT / 2);
        const uint32_t off = (uint32_t)(r * 32 + (boff & ~15)) ^ ((uint32_t)((r >> 2) & 1) << 4);
        const uint8_t* wsrc = smem + L::W_OFF + ws * L::WB + off + (boff & 15);
        uint32_t u[kEPT / 8];
        if constexpr (kEPT == 64) {  // the whole 32-byte row: both 16-byte pieces (swizzle: bit 4 ^= bit 7)
          const uint8_t* wrow = smem + L::W_OFF + ws * L::WB + r * 32;
          const uint32_t sw = (uint32_t)((r >> 2) & 1) << 4;
          const uint4 w0 = *reinterpret_cast<const uint4*>(wrow + (0u ^ sw));
          const uint4 w1 = *reinterpret_cast<const uint4*>(wrow + (16u ^ sw));
          u[0] = w0.x; u[1] = w0.y; u[2] = w0.z; u[3] = w0.w;
          u[4] = w1.x; u[5] = w1.y; u[6] = w1.z; u[7] = w1.w;
        } else if constexpr (kEPT == 32) {
          const uint4 wv = *reinterpret_cast<const uint4*>(wsrc);
          u[0] = wv.x; u[1] = wv.y; u[2] = wv.z; u[3] = wv.w;
        } else {
          const uint2 wv = *reinterpret_cast<const uint2*>(wsrc);
          u[0] = wv.x; u[1] = wv.y;
        }
        uint32_t sp[SPC];  // scale i times 2^-120 in both bf16 halves (the codes decode times 2^120)
#pragma unroll
        for (int i = 0; i < SPC; ++i) sp[i] = tc::e4m3_bf16pair_m120(tc::prmt(sc, 0u, 0x4040u + 0x0101u * i));
        uint8_t* arow = smem + L::A_OFF + slot * L::AB + r * 128;
#pragma unroll
        for (int j = 0; j < kEPT / 8; ++j) {  // 8 codes -> four bf16 pairs -> one 16-byte chunk
          uint32_t w[4];
          tc::e2m1x8_to_bf16<true>(u[j], w);
          const uint32_t spair = sp[j >> 1];
          const uint4 o = make_uint4(tc::hmul2_bf16(w[0], spair), tc::hmul2_bf16(w[1], spair),
                                     tc::hmul2_bf16(w[2], spair), tc::hmul2_bf16(w[3], spair));
          const int ck = pt * (kEPT / 8) + j;  // 16-byte chunk of the 128-byte row, 128-byte swizzle
          *reinterpret_cast<uint4*>(arow + ((ck ^ (r & 7)) << 4)) = o;
        }
        fence_proxy_async_smem();  // the MMAs read the slot through the async proxy
        __syncwarp();
        if (lane == 0) { mbar_arrive(&afull[slot]); mbar_arrive(&wempty[ws]); }
      }
    }
  } else if (warp < kWProdWarp) {
    // ---------------------------------------------- epilogue
    const int q = warp & 3;
    const int r = q * 32 + lane;
    const uint32_t lane_base = (uint32_t)(q * 32) << 16;
    const int grp = (warp - kEpiWarp0) / 4;  // columns [CPG grp, CPG (grp + 1)) of the tile
    constexpr int CPG = BM / kEpiGroups;
    griddep_wait();
    const float gsc = *reinterpret_cast<const float*>(p.scales + p.g_off);
    int n_it = 0;
    for (int it = blockIdx.x; it < total; it += gridDim.x, ++n_it) {
      const int nt = it % p.ntiles, mt = it / p.ntiles;
      const int64_t n = (int64_t)nt * kRows + r;
      const bool row_ok = n < p.N;
      const float bval = (p.bias && row_ok) ? bf16_bits_to_f32(p.bias[n]) : 0.0f;
      const int buf = n_it % L::NDB;
      if (!mbar_wait(&dfull[buf], (n_it / L::NDB) & 1, abort_flag)) break;
      tc_fence_after();
      {
        const int64_t m0 = (int64_t)mt * BM + grp * CPG;
        const uint32_t dcol = buf * BM + grp * CPG;
        uint16_t* ystage = reinterpret_cast<uint16_t*>(smem + L::Y_OFF) + grp * 16 * kRows;
#pragma unroll 1
        for (int c1 = 0; c1 < CPG; c1 += 32) {
          float acc[2][16];
          tmem_ld16(tmem_base + lane_base + dcol + c1, acc[0]);
          tmem_ld16(tmem_base + lane_base + dcol + c1 + 16, acc[1]);
          tc_wait_ld();
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {
            const int64_t mm = m0 + c1 + 16 * hh;
            if (!p.out_f32) {
              if (grp == 0)
                store_slab<0>(acc[hh], gsc, bval, r, ystage, p.y, p.M, p.N, mm, (int64_t)nt * kRows);
              else
                store_slab<1>(acc[hh], gsc, bval, r, ystage, p.y, p.M, p.N, mm, (int64_t)nt * kRows);
            } else if (row_ok) {
#pragma unroll
              for (int j = 0; j < 16; ++j)
                if (mm + j < p.M)
                  reinterpret_cast<float*>(p.y)[(mm + j) * p.N + n] = __fadd_rn(__fmul_rn(acc[hh][j], gsc), bval);
            }
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&dempty[buf]);
    }
  } else {
    // ---------------------------------------------- TMA producer: weight codes (static under programmatic
    // dependent launch, so no dependency wait)
    if (lane == 0) {
      prefetch_tmap(&maps.w);
      int g = 0;
      bool ok = true;
      for (int it = blockIdx.x; it < total && ok; it += gridDim.x) {
        const int nt = it % p.ntiles;
        for (int c = 0; c < nch; ++c, ++g) {
          const int ws = g % L::WSTAGES;
          if (g >= L::WSTAGES && !mbar_wait(&wempty[ws], ((g / L::WSTAGES) & 1) ^ 1, abort_flag)) { ok = false; break; }
          mbar_arrive_expect_tx(&wfull[ws], L::WB);
          tma_load_2d(smem + L::W_OFF + ws * L::WB, &maps.w, &wfull[ws], c * (kKC / 2), nt * kRows);
        }
      }
      if (!ok)
        for (int c = g - L::WSTAGES < 0 ? 0 : g - L::WSTAGES; c < g; ++c)
          wait_quiet(&wfull[c % L::WSTAGES], (c / L::WSTAGES) & 1);
    }
  }

  // Teardown: an mbarrier counts every warp, then warp 1 waits for the MMA issuer's last commit and
  // releases TMEM (bounded, and not cut short by the abort flag).
  tc_fence_before();
  __syncwarp();
  if (lane == 0) mbar_arrive(done);
  if (warp == 1) {
    wait_quiet(done, 0);
    if (*abort_flag) wait_quiet(drain, 0);  // else the epilogue saw every MMA finish
    tc_fence_after();
    tmem_dealloc(tmem_base, L::TMEM_COLS);
  }
}

int num_sms_w16() {
  static int n = 0;
  static std::once_flag once;
  std::call_once(once, [] {
    int dev = 0;
    cudaGetDevice(&dev);
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) n = 148;
  });
  return n;
}

template <int BM>
int launch_w4a16(const LinearArgs& a, cudaStream_t s) {
  using L = Lay16<BM>;
  auto kern = wq_w4a16_kernel<BM>;
  static std::once_flag once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(once, [&] {
    attr_err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::TOTAL);
  });
  if (attr_err != cudaSuccess) return WQ_ERR_CUDA;
  alignas(64) W16Maps maps;
  const uint64_t kb = (uint64_t)a.K / 2;
  if (!encode_tmap_2d(&maps.x, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, a.x, (uint64_t)a.K, (uint64_t)a.M,
                      (uint64_t)a.K * 2, kKC, BM, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !encode_tmap_2d(&maps.w, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.packed, kb, (uint64_t)a.N, kb, kKC / 2, kRows,
                      CU_TENSOR_MAP_SWIZZLE_32B))
    return WQ_ERR_CUDA;
  W16Params p;
  p.scales = a.scales;
  p.bias = a.bias;
  p.y = a.y;
  p.M = (int)a.M;
  p.N = (int)a.N;
  p.K = (int)a.K;
  p.ntiles = (int)((a.N + kRows - 1) / kRows);
  p.mtiles = (int)((a.M + BM - 1) / BM);
  p.total_items = p.ntiles * p.mtiles;
  p.out_f32 = a.out_f32 ? 1 : 0;
  p.weights_static = a.weights_static ? 1 : 0;
  p.g_off = (uint32_t)scales_layout(WQ_NVFP4, a.N, a.K).g_off;

  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)std::min(p.total_items, num_sms_w16()), 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = L::TOTAL;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  cfg.numAttrs = 0;
  if (a.weights_static) {
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
  }
  const cudaError_t e = cudaLaunchKernelEx(&cfg, kern, maps, p);
  count_launch();
  return e == cudaSuccess ? WQ_OK : WQ_ERR_CUDA;
}

}  // namespace

// 128-row tiles: at least this many activation rows and items, rows of at most kMaxK128 (else the
// persistent kernel: 1500 x 1280 x 5120 48.1 against 41.5 us; 1500 x 1280 x 1280 19.4 against 21.0)
constexpr int64_t kMinM128 = 512;
constexpr int64_t kMaxK128 = 2048;
constexpr int64_t kMinItems128 = 96;

int linear_w4a16_tc(const LinearArgs& a, cudaStream_t s, int* rc) {
  // NVFP4 weights, bf16 activations, one dense output; rows of whole 64-element chunks
  if (a.fmt != WQ_NVFP4 || a.M <= 16 || a.K % kKC != 0 || a.K < kKC) return 0;
  if (a.M > 0x7FFFFFFF || a.N > 0x7FFFFFFF || a.K > 0x7FFFFFFF || ((uintptr_t)a.x & 15u) != 0) return 0;
  const int64_t ntiles = (a.N + kRows - 1) / kRows;
  if (ntiles * ((a.M + 255) / 256) >= num_sms_w16()) {
    *rc = launch_w4a16<256>(a, s);
    return 1;
  }
  // fewer 256-row tiles than SMs: 128-row tiles, where they give most SMs an item
  if (a.M >= kMinM128 && a.K <= kMaxK128 && ntiles * ((a.M + 127) / 128) >= kMinItems128) {
    *rc = launch_w4a16<128>(a, s);
    return 1;
  }
  return 0;
}

int take_status_w4a16() {
  int v = 0, zero = 0;
  if (cudaMemcpyFromSymbol(&v, g_status, sizeof(int)) != cudaSuccess) return WQ_ERR_CUDA;
  cudaMemcpyToSymbol(g_status, &zero, sizeof(int));
  return v;
}

}  // namespace wq
