// wq_tcp.cu -- persistent tensor-core fused dequantise-and-multiply over a work
// list of (Linear, 128-row weight tile, BN-row activation tile) items.
//
// Serves two calls:
//   * wq_linear for M > 16 (encoder-sized activations, e.g. 1500 frames per
//     30 s window): one problem, items = n-tiles x m-tiles;
//   * wq_linear_grouped: many independent Linears of one format in ONE launch
//     (the fused Q/K/V projection of PR "Run quantized Whisper on the fused
//     Metal decode path", "Summary", generalised to any set of Linears whose
//     inputs are ready), so that the weight stream of every Linear in the group
//     shares one pipeline instead of paying a kernel boundary each.
//
// Per CTA (one per SM, persistent), warp-specialised:
//   warp 0      TMA producer: packed weight tile [128 x 64 codes] and x tile
//               [BN x 64] (128-byte swizzle) per K chunk, STAGES-deep ring.
//   warp 1      TMEM owner and MMA issuer: tcgen05.mma.kind::f16, A = decoded
//               weights in TMEM, B = x in shared memory, D in TMEM, double
//               buffered across items so the epilogue of one item overlaps the
//               main loop of the next.
//   warps 2..9  dequant: two warps per TMEM lane quarter, one thread per weight
//               row and half chunk (NF4 fold mode: per whole chunk, the two warps of
//               a quarter taking alternate chunks), packed codes -> bf16 pairs ->
//               tcgen05.st into a TMEM ring of 2 to 4 A slots.
//   warps 10..13 epilogue: tcgen05.ld, x global scale (NVFP4), + bias, store y.
//   warp 14     scale stager: one item ahead, bulk-copies the tile's scale slice
//               into shared memory (NF4: also the tile's second-level scales).
// Fold mode (decode) runs four MMA issuers -- warps 1, 14, 15 and 16, one per SM
// sub-partition -- and the scale stager on warp 17.  One thread issuing N <= 64 MMAs back to back gets about
// one per 45 cycles, and far fewer when the table loads and TMEM stores of the
// dequant warps on its sub-partition queue ahead of it; the tensor pipe itself
// takes an N = 16 MMA in about 15 cycles.  Issuers 0 and 1 take the even chunks,
// 2 and 3 the odd ones (the partial-tile slot is g & 1), and within a chunk each
// issuer of the pair takes half of the scale blocks' partial tiles.
// Every item covers the whole K range, so no cross-CTA reduction is needed.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <mutex>
#include <numeric>
#include <vector>

#include "wq_device.cuh"
#include "wq_internal.h"
#include "wq_tc_common.cuh"

namespace wq {
namespace {

using namespace tc;

constexpr int kMaxItems = 2560;   // items a launch can schedule with an explicit per-CTA list

// Warp layout.  Every mode: warp 0 TMA producer, warp 1 MMA issuer, then the dequant warps
// (kDeqQ per TMEM lane quarter, each decoding 1/kDeqQ of a chunk), then four epilogue / fold
// warps.  The other modes end with the scale stager (15 warps); fold mode (decode) adds three
// MMA issuers, one on each other SM sub-partition, before the scale stager (18 warps).  Four
// dequant warps per quarter measured slower than two.
template <int MODE>
constexpr int p_deq_q() { return 2; }
template <int MODE>
constexpr int p_epi_warp0() { return 2 + 4 * p_deq_q<MODE>(); }
template <int MODE>
constexpr int p_scale_warp() { return p_epi_warp0<MODE>() + (MODE == 2 ? 7 : 4); }
template <int MODE>
constexpr int p_warps() { return p_scale_warp<MODE>() + 1; }
constexpr int kMaxCtas = 160;     // persistent grid: one CTA per SM (152 on GB300)
constexpr int kMaxChunks = 80;    // 64-element blocks per row: K <= 5120 on this path
constexpr int kS2Max = 48;        // NF4: s2 values a tile can touch (128 * 80 / 256 + 2) + offset

struct PLay {  // the offsets of the scales blob the kernel reads (see ScalesLayout)
  uint32_t s2_off, offset_off, g_off;
};

struct PProblem {
  const uint8_t* scales;
  const uint16_t* bias;
  void* y[WQ_OUT_MAX];      // output destinations: columns [col_end[d-1], col_end[d]) of row m at
  int ld[WQ_OUT_MAX];       // y[d] + m * ld[d] + (n - col_end[d-1]) elements
  int col_end[WQ_OUT_MAX];
  int M, N, K;
  int ntiles, mtiles;
  int item_begin;
  PLay lay;
};

// Where output column n of problem pr goes: the address of its element in row 0 and the row stride
// (elements of T).
template <typename T>
struct OutCol {
  T* p;
  int64_t ld;
};
template <typename T>
__device__ __forceinline__ OutCol<T> out_col(const PProblem& pr, int64_t n) {
  int d = 0;
#pragma unroll
  for (int i = 0; i < WQ_OUT_MAX - 1; ++i) d += (n >= pr.col_end[i]) ? 1 : 0;
  const int64_t c0 = d ? pr.col_end[d - 1] : 0;
  return OutCol<T>{reinterpret_cast<T*>(pr.y[d]) + (n - c0), (int64_t)pr.ld[d]};
}

// Store one 16-column slab of a D tile (TMEM lanes = 128 weight rows n0.., columns = 16 activation
// rows m0..) through shared memory: each thread scales and writes its 16 values into stage[m][r],
// then the threads copy the [16 x 128] bf16 slab out as 16-element runs of one output row with
// 16-byte stores.  Destination boundaries are multiples of 16 columns, so a run never straddles two.
// `oc` is the destination of this thread's copy column n0 + (r % 8) * 16, resolved once per tile.
__device__ __forceinline__ void store_slab_dest(const float (&acc)[16], float gsc, float bval, int r,
                                                uint16_t* stage, const PProblem& pr, const OutCol<uint16_t>& oc,
                                                int64_t m0, int64_t n0) {
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    const float v = __fadd_rn(__fmul_rn(acc[j], gsc), bval);
    stage[j * 128 + r] = __bfloat16_as_ushort(__float2bfloat16_rn(v));
  }
  epi_bar();
  const int row = r >> 3, seg = (r & 7) * 16;
  const int64_t m = m0 + row, n = n0 + seg;
  if (m < pr.M && n < pr.N) {
    uint16_t* dst = oc.p + m * oc.ld;
    const uint16_t* src = stage + row * 128 + seg;
    if (n + 16 <= pr.N && ((uintptr_t)dst & 15u) == 0) {
      const uint4* s4 = reinterpret_cast<const uint4*>(src);
      uint4* d4 = reinterpret_cast<uint4*>(dst);
      d4[0] = s4[0];
      d4[1] = s4[1];
    } else {
      for (int e = 0; e < 16 && n + e < pr.N; ++e) dst[e] = src[e];
    }
  }
}

struct PParams {
  int nprob, total_items, out_f32, weights_static;
  int sc_bytes;    // bytes per scale buffer (max over the problems)
  int use_list;    // 1: CTA b runs items list[begin[b] .. begin[b+1]); 0: items b, b + grid, ...
  PProblem prob[kGroupMax];
  uint16_t begin[kMaxCtas + 1];
  uint32_t list[kMaxItems];  // packed item coordinates: problem | n-tile << 6 | m-tile << 19
};

struct ItemCoord {
  int p, nt, mt;
};

// The items a CTA runs, in order.
struct ItemIter {
  int pos, end, step;
  bool list;
  __device__ ItemIter(const PParams& P) {
    list = P.use_list != 0;
    if (list) { pos = P.begin[blockIdx.x]; end = P.begin[blockIdx.x + 1]; step = 1; }
    else { pos = blockIdx.x; end = P.total_items; step = gridDim.x; }
  }
  __device__ bool more() const { return pos < end; }
  __device__ void next() { pos += step; }
  __device__ ItemCoord coord(const PParams& P) const;
};

struct PMaps {
  CUtensorMap w[kGroupMax];
  CUtensorMap x[kGroupMax];
};
static_assert(sizeof(PMaps) + sizeof(PParams) <= 32000, "kernel parameter space");

// TMEM A ring slots.  NF4 decode (fold mode, 64-blocks) fits a third 256-element slot
// next to its partial-tile ring (3 x 128 + 2 x 4 x 16 = 512 columns), which lets the
// dequant warps run a chunk further ahead of the MMAs.
template <int KC, int FMT, int MODE>
constexpr int a_slots() { return KC == 256 ? ((MODE == 2 && FMT == WQ_NF4) ? 3 : 2) : 4; }

// Where the per-block weight scales are applied:
//   kScaleF32   dequant warps multiply each code's value by its block scale in fp32
//               (byte -> float pair table) -- the encoder GEMM path
//   kScaleBF16  dequant warps multiply in bf16 pairs, exact for NVFP4 only
//               (byte -> bf16 pair table) -- NVFP4 decode
//   kScaleFold  dequant warps emit unscaled values (byte -> bf16 pair table); every
//               MMA K step of a scale block writes its own TMEM partial and four fold
//               warps add  scale * partial  in fp32 -- NF4 / q4_0 / q8_0 decode
enum { kScaleF32 = 0, kScaleBF16 = 1, kScaleFold = 2 };

// KC: K elements per pipeline chunk (64 or 128: one or two 128-byte swizzle rows of x)
// Bounded wait that neither looks at the abort flag nor records a status: used after an abort, for
// the asynchronous copies and MMAs already issued to finish before the CTA releases its memory.
__device__ __forceinline__ void wait_quiet(uint64_t* bar, uint32_t parity) {
  for (uint32_t i = 0; i < kSpinLimit && !mbar_try_wait(bar, parity); ++i) {
  }
}

template <int BN, int STAGES, int FMT, int KC, int LUTREP, int MODE>
struct PSmem {
  static constexpr int SUB = KC / 64;
  static constexpr int XB = SUB * BN * 128;
  static constexpr int WB = kRows * Fmt<FMT>::WB * SUB;
  static constexpr int X_OFF = 0;
  static constexpr int W_OFF = X_OFF + STAGES * XB;
  static constexpr int LUT_OFF = W_OFF + STAGES * WB;
  static constexpr int LUT_BYTES = (FMT == WQ_Q8_0 || LUTREP == 0) ? 0 : 256 * (MODE == kScaleF32 ? 8 : 4) * LUTREP;
  static constexpr int BAR_OFF = LUT_OFF + LUT_BYTES;
  static constexpr int NBAR = 3 * STAGES + 2 * a_slots<KC, FMT, MODE>() + 9;
  static constexpr int MISC_OFF = BAR_OFF + NBAR * 8;
  static constexpr int Y_OFF = (MISC_OFF + 16 + 127) / 128 * 128;             // [2] 4 KB output slabs
  static constexpr int S2_OFF = Y_OFF + 2 * 16 * kRows * 2;                   // [2][kS2Max] NF4 s2 + offset
  static constexpr int SC_OFF = (S2_OFF + 2 * kS2Max * 4 + 127) / 128 * 128;  // [2] raw scale slices
  static constexpr int FIXED = SC_OFF + 1024;                                   // + alignment slack
  // one tile's scale bytes as stored in the blob (row-major): 4 bytes per row per
  // 64-block (NVFP4 / q4_0 / q8_0), 1 byte (NF4); two buffers
  static constexpr int sc_bytes(int blocks) { return blocks * kRows * Fmt<FMT>::SCB; }
  static constexpr int total(int blocks) { return FIXED + 2 * sc_bytes(blocks); }
  // the longest K (in 64-blocks) whose scale slices fit next to the pipeline
  static constexpr int max_blocks() {
    const int fit = Fmt<FMT>::SCB == 0 ? kMaxChunks : (227 * 1024 - FIXED) / (2 * kRows * Fmt<FMT>::SCB);
    return fit < kMaxChunks ? fit : kMaxChunks;
  }
  static_assert(max_blocks() >= 20, "shared memory budget: K = 1280 must fit");
};

template <int FMT>
constexpr int scale_groups_per_128() { return FMT == WQ_NF4 ? 2 : FMT == WQ_NVFP4 ? 8 : 4; }

template <int BN, int KC, int FMT, int MODE>
struct PTmem {
  static constexpr int NA = a_slots<KC, FMT, MODE>();
  static constexpr int ACOLS = KC / 2;  // 32-bit columns per A slot (bf16 pairs)
  static constexpr int D_COL = NA * ACOLS;
  // kScaleFold: a double-buffered ring of per-scale-block partial tiles instead of D
  static constexpr int G = scale_groups_per_128<FMT>() * KC / 128;
  // accumulator buffers: two (epilogue overlaps the next item) when they fit next to the A ring
  static constexpr int NDB = (MODE == kScaleFold || D_COL + 2 * BN <= 512) ? 2 : 1;
  static constexpr int USED = D_COL + NDB * BN * (MODE == kScaleFold ? G : 1);
  static constexpr int ALLOC = USED <= 256 ? 256 : 512;
  static_assert(USED <= 512, "TMEM budget");
};

__device__ __forceinline__ ItemCoord item_coord(const PParams& P, int i) {
  int p = 0;
  while (p + 1 < P.nprob && P.prob[p + 1].item_begin <= i) ++p;
  const int local = i - P.prob[p].item_begin;
  const int nt_count = P.prob[p].ntiles;
  return ItemCoord{p, local % nt_count, local / nt_count};
}

__device__ __forceinline__ ItemCoord ItemIter::coord(const PParams& P) const {
  if (list) {
    const uint32_t v = P.list[pos];
    return ItemCoord{(int)(v & 63u), (int)((v >> 6) & 8191u), (int)(v >> 19)};
  }
  return item_coord(P, pos);
}

template <int BN, int STAGES, int FMT, int KC, int LUTREP, int MODE>
__global__ void __launch_bounds__(p_warps<MODE>() * 32, 1)
    wq_tcp_kernel(const __grid_constant__ PMaps maps, const __grid_constant__ PParams P) {
  using S = PSmem<BN, STAGES, FMT, KC, LUTREP, MODE>;
  using T = PTmem<BN, KC, FMT, MODE>;
  static_assert(MODE != kScaleFold || (BN == 16 && FMT != WQ_NVFP4), "fold mode: decode tiles");
  static_assert(MODE != kScaleBF16 || FMT == WQ_NVFP4 || FMT == WQ_FP8, "bf16 scaling is exact for NVFP4 only");
  static_assert(LUTREP != 0 || ((FMT == WQ_NVFP4 || FMT == WQ_FP8) && MODE == kScaleBF16),
                "register decode: NVFP4, FP8");
  constexpr bool FOLD = MODE == kScaleFold;
  constexpr int kNA = T::NA;
  // fold warps read chunk g's partials once A slot g % NA is released, and the partial
  // ring is indexed g & 1: the two rings must coincide
  // the partial-tile ring has two slots (g & 1) whatever the A ring's depth
  constexpr int kDeqQ = p_deq_q<MODE>();
  constexpr int kDeqWarps = 4 * kDeqQ;
  // NF4 fold mode: the kDeqQ warps of a lane quarter take whole chunks in turn (kDeqG groups, chunk g
  // to group g % kDeqG); else each decodes 1/kDeqQ of every chunk (q4_0 decode measured 11 % slower
  // in turns)
  constexpr int kDeqG = (FOLD && FMT == WQ_NF4) ? kDeqQ : 1;
  constexpr int kDeqPart = kDeqQ / kDeqG;  // parts of a chunk
  constexpr int kGroupWarps = kDeqWarps / kDeqG;
  constexpr int kEpiWarp0 = p_epi_warp0<MODE>();
  constexpr int SCALE_CONSUMERS = FOLD ? 4 : kDeqWarps;
  constexpr int NWARPS = p_warps<MODE>();
  constexpr int SCALE_WARP = p_scale_warp<MODE>();
  constexpr int NISSUE = FOLD ? 4 : 1;  // MMA issuers; fold mode: two per chunk
  constexpr int CHUNK_COMMITS = FOLD ? 2 : 1;
  constexpr int SUB = S::SUB;
  constexpr int NE = KC / kDeqPart;  // elements of a row each dequant warp decodes per chunk
  static_assert(NE == 32 || NE % 64 == 0, "a dequant warp decodes half a 64-block or whole blocks");
  constexpr uint32_t IDESC = idesc_bf16(kRows, BN);
  constexpr int WCHUNK = Fmt<FMT>::WB * SUB;  // packed bytes of one row per chunk
  // row bytes of one W TMA box: the swizzle width, or (80-byte units) the whole unswizzled chunk
  constexpr int WRB = Fmt<FMT>::UNIT ? WCHUNK : (WCHUNK < 128 ? WCHUNK : 128);
  static_assert(!Fmt<FMT>::UNIT || (KC == 128 && MODE == kScaleF32), "unit formats: GEMM tiles of one unit");
  constexpr int WNBOX = WCHUNK / WRB;

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + S::BAR_OFF);
  uint64_t* wfull = bars;           // [STAGES] a stage's weight tile has landed
  uint64_t* empty = bars + STAGES;
  uint64_t* afull = bars + 2 * STAGES;
  uint64_t* aempty = afull + kNA;
  uint64_t* dfull = aempty + kNA;  // [2]
  uint64_t* dempty = dfull + 2;    // [2]
  uint64_t* sfull = dempty + 2;    // [2]
  uint64_t* sempty = sfull + 2;    // [2]
  uint64_t* done = sempty + 2;     // every warp has finished (TMEM may be released)
  uint64_t* xfull = done + 1;      // [STAGES] a stage's activation tile has landed
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + S::MISC_OFF);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + S::MISC_OFF + 4);
  // after an abort, every MMA issuer's last commit (all MMAs finished); in the 16-byte misc block
  static_assert(S::MISC_OFF % 8 == 0, "mbarrier alignment");
  uint64_t* drain = reinterpret_cast<uint64_t*>(smem + S::MISC_OFF + 8);
  float2* lut = reinterpret_cast<float2*>(smem + S::LUT_OFF);
  uint32_t* lut32 = reinterpret_cast<uint32_t*>(smem + S::LUT_OFF);
  uint8_t* scbuf = smem + S::SC_OFF;
  float* s2buf = reinterpret_cast<float*>(smem + S::S2_OFF);

  const int warp = (int)warp_id(), lane = (int)lane_id();
  // MMA issuer index: warp 1 -> 0; fold mode also warps 14, 15, 16 -> 1, 2, 3
  const int issuer =
      (warp == 1) ? 0 : (FOLD && warp >= kEpiWarp0 + 4 && warp <= kEpiWarp0 + 6) ? warp - (kEpiWarp0 + 3) : -1;

  if (threadIdx.x == 0) {
    for (int i = 0; i < STAGES; ++i) {
      mbar_init(&wfull[i], 1);
      mbar_init(&xfull[i], 1);
      mbar_init(&empty[i], CHUNK_COMMITS + kGroupWarps);
    }
    for (int i = 0; i < kNA; ++i) { mbar_init(&afull[i], kGroupWarps); mbar_init(&aempty[i], CHUNK_COMMITS); }
    mbar_init(done, NWARPS);
    mbar_init(drain, NISSUE);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&dfull[i], 1);   // kScaleFold: a partial-tile slot is full
      mbar_init(&dempty[i], 4);  // kScaleFold: a partial-tile slot was folded
      mbar_init(&sfull[i], 32);
      mbar_init(&sempty[i], SCALE_CONSUMERS);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (FMT != WQ_Q8_0 && LUTREP > 0) {
    for (int i = threadIdx.x; i < 256 * LUTREP; i += NWARPS * 32) {
      const uint32_t b = (uint32_t)(i / LUTREP);
      if (MODE == kScaleF32)
        lut[i] = make_float2(nibble_value<FMT>(b & 15u), nibble_value<FMT>(b >> 4));
      else
        lut32[i] = nibble_pair_bf16<FMT>(b);
    }
  }
  if (warp == 1) tmem_alloc(tmem_slot, T::ALLOC);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  griddep_launch_dependents();

  const int total = P.total_items;
  if (warp == 0) {
    // ------------------------------------------------ TMA producer
    if (lane == 0) {
      for (int i = 0; i < P.nprob; ++i) {
        prefetch_tmap(&maps.w[i]);
        prefetch_tmap(&maps.x[i]);
      }
      // weights of the first STAGES chunks may stream (and be decoded) before the preceding
      // kernel finishes; weights and activations have separate barriers, so only the MMAs
      // wait for the activations
      int pre = 0;
      if (P.weights_static) {
        int g = 0;
        for (ItemIter ii(P); ii.more() && g < STAGES; ii.next()) {
          const ItemCoord ic = ii.coord(P);
          const int nch = (P.prob[ic.p].K + KC - 1) / KC;
          for (int c = 0; c < nch && g < STAGES; ++c, ++g) {
            mbar_arrive_expect_tx(&wfull[g], (uint32_t)S::WB);
            for (int b = 0; b < WNBOX; ++b)
              tma_load_2d(smem + S::W_OFF + g * S::WB + b * 128 * WRB, &maps.w[ic.p], &wfull[g],
                          c * WCHUNK + b * WRB, ic.nt * kRows);
          }
        }
        pre = g;
      }
      griddep_wait();
      int g = 0;
      bool ok = true;
      for (ItemIter ii(P); ii.more() && ok; ii.next()) {
        const ItemCoord ic = ii.coord(P);
        const int nch = (P.prob[ic.p].K + KC - 1) / KC;
        for (int c = 0; c < nch; ++c, ++g) {
          const int s = g % STAGES;
          if (g >= pre) {
            // stage s is free once chunk g - STAGES is consumed (x by its MMAs, weights by the
            // dequant warps); a per-stage barrier cannot complete twice before this wait
            if (g >= STAGES && !mbar_wait(&empty[s], ((g / STAGES) & 1) ^ 1, abort_flag)) { ok = false; break; }
            mbar_arrive_expect_tx(&wfull[s], (uint32_t)S::WB);
            for (int b = 0; b < WNBOX; ++b)
              tma_load_2d(smem + S::W_OFF + s * S::WB + b * 128 * WRB, &maps.w[ic.p], &wfull[s],
                          c * WCHUNK + b * WRB, ic.nt * kRows);
          }
          mbar_arrive_expect_tx(&xfull[s], (uint32_t)S::XB);
#pragma unroll
          for (int j = 0; j < SUB; ++j)
            tma_load_2d(smem + S::X_OFF + s * S::XB + j * BN * 128, &maps.x[ic.p], &xfull[s], c * KC + j * 64,
                        ic.mt * BN);
        }
      }
      // stopped by a wait that ran out: let the copies of the stages in flight land before exit
      if (!ok)
        for (int c = g - STAGES < 0 ? 0 : g - STAGES; c < g; ++c) {
          wait_quiet(&wfull[c % STAGES], (c / STAGES) & 1);
          wait_quiet(&xfull[c % STAGES], (c / STAGES) & 1);
        }
    }
  } else if (issuer >= 0) {
    // ------------------------------------------------ MMA issuers (whole warp waits, lane 0 issues)
    // Fold mode: issuers 0 and 1
    // take the even chunks, 2 and 3 the odd ones, and each issuer of a pair the partial tiles
    // of half of the chunk's scale blocks; a commit tracks only its own thread's MMAs, so the
    // A-slot and stage barriers expect one commit from each issuer of the pair.
    const int pair = issuer >> 1, half = issuer & 1;
    const uint64_t xdesc0 = smem_desc(smem_u32(smem + S::X_OFF), 16, 1024, 2);
    int g = 0, n_it = 0;
    bool ok = true;
    for (ItemIter ii(P); ii.more() && ok; ii.next(), ++n_it) {
      const ItemCoord ic = ii.coord(P);
      const int nch = (P.prob[ic.p].K + KC - 1) / KC;
      const int buf = n_it % T::NDB;
      if (!FOLD && !mbar_wait_lanes(&dempty[buf], ((n_it / T::NDB) & 1) ^ 1, lane == 0 && n_it >= T::NDB,
                                    abort_flag))
        break;
      tc_fence_after();
      const uint32_t d_tmem = tmem_base + T::D_COL + buf * BN;
      for (int c = 0; c < nch; ++c, ++g) {
        if (FOLD && (g & 1) != pair) continue;
        const int s = g % STAGES, slot = g % kNA;
        // lane 0: the A slot; lane 1 (fold mode): the partial-tile slot; lane 2: the x tile
        uint64_t* wb = (lane == 0) ? &afull[slot] : (lane == 1) ? &dempty[g & 1] : &xfull[s];
        const uint32_t wp = (lane == 0) ? ((g / kNA) & 1) : (lane == 1) ? (((g >> 1) & 1) ^ 1) : ((g / STAGES) & 1);
        const bool act = (lane == 0) || (FOLD && lane == 1 && g >= 2) || (lane == 2);
        if (!mbar_wait_lanes(wb, wp, act, abort_flag)) { ok = false; break; }
        tc_fence_after();
        if (lane == 0) {
          // descriptors as base + compile-time offsets (the 14-bit address field cannot
          // carry: shared addresses stay below 2^18)
          const uint64_t xdesc = xdesc0 + (uint64_t)((s * S::XB) >> 4);
          const uint32_t a_tmem = tmem_base + slot * T::ACOLS;
          if (FOLD) {
            constexpr int KPG = (KC / 16) / T::G;  // MMA K steps per scale block
            constexpr int GH = T::G / 2;           // scale blocks per issuer
            const uint32_t p_tmem = tmem_base + T::D_COL + ((g & 1) * T::G + half * GH) * BN;
#pragma unroll
            for (int step = 0; step < KPG; ++step)
#pragma unroll
              for (int gg = 0; gg < GH; ++gg) {
                // consecutive MMAs go to different scale blocks' partial tiles
                const int kk = (half * GH + gg) * KPG + step;
                mma_bf16_ts(p_tmem + gg * BN, a_tmem + kk * 8, xdesc + (uint64_t)((kk / 4) * BN * 8 + (kk % 4) * 2),
                            IDESC, step != 0 ? 1u : 0u);
              }
          } else {
#pragma unroll
            for (int kk = 0; kk < KC / 16; ++kk)
              mma_bf16_ts(d_tmem, a_tmem + kk * 8, xdesc + (uint64_t)((kk / 4) * BN * 8 + (kk % 4) * 2), IDESC,
                          (c | kk) != 0 ? 1u : 0u);
          }
          tc_commit(&aempty[slot]);
          tc_commit(&empty[s]);
        }
        __syncwarp();
      }
      if (ok && !FOLD && lane == 0) tc_commit(&dfull[buf]);
      __syncwarp();
    }
    // after an abort: a commit that tracks every MMA this thread issued, for the teardown's wait
    if (lane == 0 && (!ok || *abort_flag)) tc_commit(drain);
  } else if (warp < kEpiWarp0) {
    // ------------------------------------------------ dequant warps: half h of every chunk
    const int q = warp & 3;
    const int h = kDeqG > 1 ? 0 : (warp - 2) / 4;    // which 1/kDeqPart of the chunk
    const int grp = kDeqG > 1 ? (warp - 2) / 4 : 0;  // chunks g with g % kDeqG == grp
    const int r = q * 32 + lane;
    const int lsel = (LUTREP > 1) ? (lane & (LUTREP - 1)) : 0;
    const uint32_t lane_base = (uint32_t)(q * 32) << 16;
    int g = 0, n_it = 0;
    bool ok = true;
    for (ItemIter ii(P); ii.more() && ok; ii.next(), ++n_it) {
      const ItemCoord ic = ii.coord(P);
      const PProblem& pr = P.prob[ic.p];
      const int nb = pr.K / 64;                 // 64-element blocks per row
      const int nch = (pr.K + KC - 1) / KC;
      const int sb = n_it & 1;
      const int64_t n = (int64_t)ic.nt * kRows + r;
      const bool row_ok = n < pr.N;
      if (!FOLD && !mbar_wait(&sfull[sb], (n_it >> 1) & 1, abort_flag)) break;
      const uint8_t* sc = scbuf + sb * P.sc_bytes;
      const float* s2s = s2buf + sb * kS2Max;
      const int64_t g0 = ((int64_t)ic.nt * kRows * nb) / 256;  // NF4: first s2 group of the tile
      const float off = (FMT == WQ_NF4 && !FOLD) ? s2s[kS2Max - 1] : 0.0f;
      for (int c = 0; c < nch; ++c, ++g) {
        if (kDeqG > 1 && g % kDeqG != grp) continue;  // another group's chunk
        const int s = g % STAGES, slot = g % kNA;
        constexpr int NBW = (NE >= 64) ? NE / 64 : 1;  // 64-blocks (or half of one) this warp decodes
        uint32_t sword[NBW];
#pragma unroll
        for (int bb = 0; bb < NBW; ++bb) {
          // the 64-block this warp decodes (NE >= 64), or the block holding its half (NE == 32)
          const int blk = (NE >= 64) ? (KC / 64) * c + NBW * h + bb : (KC / 64) * c + h / 2;
          sword[bb] = 0u;
          if (!FOLD && Fmt<FMT>::SCB != 0 && row_ok && blk < nb) {
            if (FMT == WQ_NF4) {
              const int8_t qa = (int8_t)sc[r * nb + blk];
              const float s2 = s2s[(n * nb + blk) / 256 - g0];
              sword[bb] = __float_as_uint(__fadd_rn(__fmul_rn((float)qa, s2), off));
            } else {
              sword[bb] = *reinterpret_cast<const uint32_t*>(sc + 4 * (r * nb + blk));
            }
          }
        }
        if (!mbar_wait(&wfull[s], (g / STAGES) & 1, abort_flag)) { ok = false; break; }
        if (g >= kNA && !mbar_wait(&aempty[slot], ((g / kNA) & 1) ^ 1, abort_flag)) { ok = false; break; }
        const uint8_t* wstage = smem + S::W_OFF + s * S::WB;
        constexpr int NES = NE / NBW;                          // elements per decode call (32 or 64)
        constexpr int CPS = NES / (Fmt<FMT>::BYTE ? 16 : 32);  // 16-byte chunks per call
        const int ck0 = h * (WCHUNK / (16 * kDeqPart));         // first 16-byte chunk of this warp's part
#pragma unroll (kDeqG > 1 ? 1 : NBW)  // whole chunks: one 64-block at a time (no register spills)
        for (int bb = 0; bb < NBW; ++bb) {
          uint32_t v[NES / 2];
          if constexpr (Fmt<FMT>::UNIT) {
            // one unit per chunk (KC = 128): this warp's 64 elements are nibble bytes [32h, 32h + 32)
            // and side bytes [64 + 8h, 72 + 8h) of row r's unit
            static_assert(NES == 64 && NBW == 1, "unit decode");
            const uint8_t* rowp = wstage + r * WCHUNK;
            const uint4 nibv[2] = {*reinterpret_cast<const uint4*>(rowp + 32 * h),
                                   *reinterpret_cast<const uint4*>(rowp + 32 * h + 16)};
            const uint2 side = *reinterpret_cast<const uint2*>(rowp + 64 + 8 * h);
            decode_unit64<FMT, LUTREP>(nibv, side, sword[bb], lut, lsel, v);
            tmem_st_n(tmem_base + lane_base + slot * T::ACOLS + h * (NE / 2) + bb * (NES / 2), v);
            continue;
          }
          uint4 wv[CPS];
#pragma unroll
          for (int k = 0; k < CPS; ++k) wv[k] = load_wchunk<WRB, WNBOX>(wstage, r, ck0 + bb * CPS + k);
          const int part = (NE == 32) ? (h & 1) : 0;
          if constexpr (FMT == WQ_FP8)
            decode_span_fp8<NES>(wv, v);
          else if constexpr (LUTREP == 0)
            decode_span_nvfp4_reg<NES>(sword[bb], part, wv, v);
          else if constexpr (MODE == kScaleF32)
            decode_span<FMT, NES, LUTREP>(sword[bb], part, wv, lut, lsel, v);
          else
            decode_span_bf16<FMT, NES, LUTREP, MODE == kScaleBF16>(sword[bb], part, wv, lut32, lsel, v);
          tmem_st_n(tmem_base + lane_base + slot * T::ACOLS + h * (NE / 2) + bb * (NES / 2), v);
        }
        tc_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) { mbar_arrive(&afull[slot]); mbar_arrive(&empty[s]); }
      }
      __syncwarp();
      if (!FOLD && lane == 0) mbar_arrive(&sempty[sb]);
    }
  } else if (warp < kEpiWarp0 + 4) {
    // ------------------------------------------------ epilogue warps
    const int q = warp & 3;
    const int r = q * 32 + lane;
    const uint32_t lane_base = (uint32_t)(q * 32) << 16;
    griddep_wait();
    int n_it = 0, g = 0;
    for (ItemIter ii(P); ii.more(); ii.next(), ++n_it) {
      const ItemCoord ic = ii.coord(P);
      const PProblem& pr = P.prob[ic.p];
      const int buf = n_it % T::NDB;
      const int64_t n = (int64_t)ic.nt * kRows + r;
      const bool row_ok = n < pr.N;
      // NVFP4: the tensor's global scale; FP8: the row's scale (0 past the last row)
      const float gsc = (FMT == WQ_NVFP4) ? *reinterpret_cast<const float*>(pr.scales + pr.lay.g_off)
                        : (FMT == WQ_FP8) ? (row_ok ? reinterpret_cast<const float*>(pr.scales)[n] : 0.0f)
                                          : 1.0f;
      const float bval = (pr.bias && row_ok) ? bf16_bits_to_f32(pr.bias[n]) : 0.0f;
      const int m0 = ic.mt * BN;
      if (FOLD) {
        // fold the per-scale-block partial tiles of every chunk: acc += scale * partial
        const int nb = pr.K / 64;
        const int nch = (pr.K + KC - 1) / KC;
        const int sb = n_it & 1;
        if (!mbar_wait(&sfull[sb], (n_it >> 1) & 1, abort_flag)) break;
        const uint8_t* sc = scbuf + sb * P.sc_bytes;
        const float* s2s = s2buf + sb * kS2Max;
        const int64_t g0 = ((int64_t)ic.nt * kRows * nb) / 256;
        const float off = (FMT == WQ_NF4) ? s2s[kS2Max - 1] : 0.0f;
        float acc[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) acc[j] = 0.0f;
        bool ok = true;
        for (int c = 0; c < nch; ++c, ++g) {
          // block scales of this row for the chunk's scale blocks (0 past the end of K)
          float sg[T::G];
#pragma unroll
          for (int grp = 0; grp < T::G; ++grp) {
            float sv = 0.0f;
            if (FMT == WQ_NF4) {
              const int blk = c * T::G + grp;  // 64-blocks
              if (row_ok && blk < nb) {
                const float s2 = s2s[(n * nb + blk) / 256 - g0];
                sv = __fadd_rn(__fmul_rn((float)(int8_t)sc[r * nb + blk], s2), off);
              }
            } else {  // q4_0 / q8_0: 32-blocks, fp16 d
              const int j32 = c * T::G + grp;
              if (row_ok && j32 < 2 * nb)
                sv = f16_bits_to_f32(*reinterpret_cast<const uint16_t*>(sc + 4 * r * nb + 2 * j32));
            }
            sg[grp] = sv;
          }
          // the partials of chunk g are complete when its MMAs release A slot g % NA (== g & 1)
          if (!mbar_wait(&aempty[g % kNA], (g / kNA) & 1, abort_flag)) { ok = false; break; }
          tc_fence_after();
#pragma unroll
          for (int grp = 0; grp < T::G; ++grp) {
            float pt[16];
            tmem_ld16(tmem_base + lane_base + T::D_COL + ((g & 1) * T::G + grp) * BN, pt);
            tc_wait_ld();
#pragma unroll
            for (int j = 0; j < 16; ++j) acc[j] = fmaf(sg[grp], pt[j], acc[j]);
          }
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&dempty[g & 1]);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&sempty[sb]);
        if (!ok) break;
        if (row_ok) {
          const OutCol<float> o32 = out_col<float>(pr, n);
          const OutCol<__nv_bfloat16> o16 = out_col<__nv_bfloat16>(pr, n);
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const int m = m0 + j;
            if (m < pr.M) {
              const float val = __fadd_rn(acc[j], bval);
              if (P.out_f32)
                o32.p[(int64_t)m * o32.ld] = val;
              else
                o16.p[(int64_t)m * o16.ld] = __float2bfloat16_rn(val);
            }
          }
        }
        continue;
      }
      if (!mbar_wait(&dfull[buf], (n_it / T::NDB) & 1, abort_flag)) break;
      tc_fence_after();
      uint16_t* ystage = reinterpret_cast<uint16_t*>(smem + S::Y_OFF);
      const int64_t n_copy = (int64_t)ic.nt * kRows + (r & 7) * 16;  // the column this thread copies out
      const OutCol<uint16_t> oc16 = out_col<uint16_t>(pr, n_copy < pr.N ? n_copy : 0);
      const OutCol<float> o32 = out_col<float>(pr, n);
#pragma unroll 1
      for (int c0 = 0; c0 < BN; c0 += 16) {
        float acc[16];
        tmem_ld16(tmem_base + lane_base + T::D_COL + buf * BN + c0, acc);
        tc_wait_ld();
        if (!P.out_f32) {
          store_slab_dest(acc, gsc, bval, r, ystage + ((c0 / 16) & 1) * 16 * kRows, pr, oc16, m0 + c0,
                          (int64_t)ic.nt * kRows);
        } else if (row_ok) {
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const int m = m0 + c0 + j;
            if (m < pr.M) o32.p[(int64_t)m * o32.ld] = __fadd_rn(__fmul_rn(acc[j], gsc), bval);
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&dempty[buf]);
    }
  } else if (warp == SCALE_WARP) {
    // ------------------------------------------------ scale warp: one item ahead of the dequant warps,
    // one bulk copy of the tile's scale slice (contiguous in the blob) into shared memory
    int n_it = 0;
    bool ok = true;
    for (ItemIter ii(P); ii.more(); ii.next(), ++n_it) {
      const ItemCoord ic = ii.coord(P);
      const PProblem& pr = P.prob[ic.p];
      const int nb = pr.K / 64;
      const int sb = n_it & 1;
      if (n_it >= 2 && !mbar_wait(&sempty[sb], ((n_it >> 1) & 1) ^ 1, abort_flag)) { ok = false; break; }
      const int64_t n0 = (int64_t)ic.nt * kRows;
      const int rows = (int)((pr.N - n0) < kRows ? (pr.N - n0) : kRows);
      const int row_bytes = Fmt<FMT>::SCB * nb;
      // 16-byte aligned source (n0 * row_bytes is a multiple of 16) and a size rounded up to 16:
      // the scale regions of the blob are zero-padded to 16 bytes, so this stays inside it
      const uint32_t bytes = (uint32_t)(((int64_t)rows * row_bytes + 15) / 16 * 16);
      if (FMT == WQ_NF4) {
        const int64_t b_lo = n0 * nb, b_hi = b_lo + (int64_t)rows * nb;  // absmax index range
        const int64_t g0 = b_lo / 256, g1 = (b_hi - 1) / 256;
        float* s2s = s2buf + sb * kS2Max;
        const float* s2g = reinterpret_cast<const float*>(pr.scales + pr.lay.s2_off);
        for (int64_t gi = g0 + lane; gi <= g1; gi += 32) s2s[gi - g0] = s2g[gi];
        if (lane == 0) s2s[kS2Max - 1] = *reinterpret_cast<const float*>(pr.scales + pr.lay.offset_off);
      }
      if (lane == 0 && bytes > 0) {
        uint64_t* bar = &sfull[sb];
        mbar_arrive_expect_tx(bar, bytes);
        const uint8_t* src = pr.scales + n0 * row_bytes;
        asm volatile(
            "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                smem_u32(scbuf + sb * P.sc_bytes)),
            "l"(src), "r"(bytes), "r"(smem_u32(bar))
            : "memory");
      } else {
        mbar_arrive(&sfull[sb]);
      }
    }
    // stopped by a wait that ran out: the scale copies of the (at most two) items in flight land
    if (!ok)
      for (int it = n_it - 2 < 0 ? 0 : n_it - 2; it < n_it; ++it) wait_quiet(&sfull[it & 1], (it >> 1) & 1);
  }

  // Teardown: every warp arrives once its own work is over (its MMAs waited for by the
  // fold / epilogue warps, its TMEM stores and loads waited for); warp 1 releases TMEM after
  // all arrivals.  An mbarrier with an explicit count, not a CTA-wide bar.sync, so that no
  // lane-divergent path of a warp-specialised role can complete it early.
  tc_fence_before();
  __syncwarp();
  if (lane == 0) mbar_arrive(done);
  if (warp == 1) {
    // bounded, and not cut short by the abort flag: every other wait is bounded, so every
    // warp arrives; the issuers' last commits mean no MMA still uses TMEM; TMEM is released in any
    // case before the CTA exits
    wait_quiet(done, 0);
    if (*abort_flag) wait_quiet(drain, 0);  // else the fold / epilogue warps saw every MMA finish
    tc_fence_after();
    tmem_dealloc(tmem_base, T::ALLOC);
  }
}

int num_sms() {
  static int n = 0;
  static std::once_flag once;
  std::call_once(once, [] {
    int dev = 0;
    cudaGetDevice(&dev);
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) n = 148;
  });
  return n;
}

template <int BN, int STAGES, int FMT, int KC, int LUTREP, int MODE>
int launch_tcp(const LinearArgs* probs, int count, bool out_f32, bool weights_static, cudaStream_t s) {
  using S = PSmem<BN, STAGES, FMT, KC, LUTREP, MODE>;
  auto kern = wq_tcp_kernel<BN, STAGES, FMT, KC, LUTREP, MODE>;
  static std::once_flag once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(once, [&] {
    attr_err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, S::total(S::max_blocks()));
  });
  if (attr_err != cudaSuccess) return WQ_ERR_CUDA;

  // heavier items (longer K) first, so the round-robin over CTAs stays balanced
  std::vector<int> order(count);
  std::iota(order.begin(), order.end(), 0);
  std::stable_sort(order.begin(), order.end(), [&](int a, int b) { return probs[a].K > probs[b].K; });

  static PMaps maps;    // host staging; copied into the launch's parameter buffer
  static PParams P;
  static std::mutex mu;
  std::lock_guard<std::mutex> lock(mu);
  P.nprob = count;
  P.out_f32 = out_f32 ? 1 : 0;
  P.weights_static = weights_static ? 1 : 0;
  int items = 0;
  for (int j = 0; j < count; ++j) {
    const LinearArgs& a = probs[order[j]];
    PProblem& pr = P.prob[j];
    pr.scales = a.scales;
    pr.bias = a.bias;
    for (int d = 0; d < WQ_OUT_MAX; ++d) {
      const int dd = d < a.nout ? d : a.nout - 1;
      pr.y[d] = a.ys[dd];
      pr.ld[d] = (int)a.ld[dd];
      pr.col_end[d] = (int)a.col_end[dd];
    }
    pr.M = (int)a.M;
    pr.N = (int)a.N;
    pr.K = (int)a.K;
    pr.ntiles = (int)((a.N + kRows - 1) / kRows);
    pr.mtiles = (int)((a.M + BN - 1) / BN);
    pr.item_begin = items;
    {
      const ScalesLayout L = scales_layout(FMT, a.N, a.K);
      pr.lay = PLay{(uint32_t)L.s2_off, (uint32_t)L.offset_off, (uint32_t)L.g_off};
    }
    items += pr.ntiles * pr.mtiles;
    const uint64_t wrow = (uint64_t)packed_row_bytes(FMT, a.K);
    if (!encode_tmap_2d(&maps.x[j], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, a.x, (uint64_t)a.K, (uint64_t)a.M,
                        (uint64_t)a.K * 2, 64, BN, CU_TENSOR_MAP_SWIZZLE_128B))
      return WQ_ERR_CUDA;
    constexpr int wbox = Fmt<FMT>::UNIT ? Fmt<FMT>::WB * (KC / 64) : std::min(Fmt<FMT>::WB * (KC / 64), 128);
    const CUtensorMapSwizzle wswz = Fmt<FMT>::UNIT ? CU_TENSOR_MAP_SWIZZLE_NONE : swizzle_of<std::min(wbox, 128)>();
    if (!encode_tmap_2d(&maps.w[j], CU_TENSOR_MAP_DATA_TYPE_UINT8, a.packed, wrow, (uint64_t)a.N, wrow, wbox, kRows,
                        wswz))
      return WQ_ERR_CUDA;
  }
  P.total_items = items;
  if (items == 0) return WQ_OK;
  const int grid = std::min(std::min(items, num_sms()), kMaxCtas);
  // longest-processing-time-first assignment of items to CTAs (cost = K chunks + a fixed
  // per-item overhead); items are visited heaviest first, each to the least-loaded CTA
  P.use_list = 1;
  if (items > kMaxItems) P.use_list = 0;
  for (int j = 0; j < count; ++j)
    if (P.prob[j].ntiles > 8191 || P.prob[j].mtiles > 8191) P.use_list = 0;
  if (P.use_list) {
    std::vector<int> order_items(items);
    std::vector<int> cost(items);
    for (int j = 0; j < count; ++j)
      for (int i = 0; i < P.prob[j].ntiles * P.prob[j].mtiles; ++i)
        cost[P.prob[j].item_begin + i] = (P.prob[j].K + KC - 1) / KC + 2;
    std::iota(order_items.begin(), order_items.end(), 0);
    std::stable_sort(order_items.begin(), order_items.end(), [&](int a, int b) { return cost[a] > cost[b]; });
    std::vector<std::vector<int>> bins(grid);
    std::vector<std::pair<long, int>> heap;  // (load, cta), min-heap
    for (int b = 0; b < grid; ++b) heap.push_back({0L, b});
    auto cmp = [](const std::pair<long, int>& a, const std::pair<long, int>& b) { return a > b; };
    std::make_heap(heap.begin(), heap.end(), cmp);
    for (int it : order_items) {
      std::pop_heap(heap.begin(), heap.end(), cmp);
      auto& top = heap.back();
      bins[top.second].push_back(it);
      top.first += cost[it];
      std::push_heap(heap.begin(), heap.end(), cmp);
    }
    std::vector<uint32_t> packed(items);
    for (int j = 0; j < count; ++j)
      for (int i = 0; i < P.prob[j].ntiles * P.prob[j].mtiles; ++i)
        packed[P.prob[j].item_begin + i] =
            (uint32_t)j | ((uint32_t)(i % P.prob[j].ntiles) << 6) | ((uint32_t)(i / P.prob[j].ntiles) << 19);
    int pos = 0;
    for (int b = 0; b < grid; ++b) {
      P.begin[b] = (uint16_t)pos;
      for (int it : bins[b]) P.list[pos++] = packed[it];
    }
    P.begin[grid] = (uint16_t)pos;
  }
  int max_blocks = 1;
  for (int j = 0; j < count; ++j) max_blocks = std::max(max_blocks, P.prob[j].K / 64);
  if (max_blocks > S::max_blocks()) return WQ_ERR_SHAPE;  // callers pick a configuration that fits
  P.sc_bytes = S::sc_bytes(max_blocks);

  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid, 1, 1);
  cfg.blockDim = dim3(p_warps<MODE>() * 32, 1, 1);
  cfg.dynamicSmemBytes = S::total(max_blocks);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  int na = 0;
  if (weights_static) {
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    na = 1;
  }
  cfg.attrs = attr;
  cfg.numAttrs = na;
  cudaError_t e = cudaLaunchKernelEx(&cfg, kern, maps, P);
  count_launch();
  return e == cudaSuccess ? WQ_OK : WQ_ERR_CUDA;
}

// decode: 256-element chunks, lane-replicated bf16-pair table, block scales folded after the
// MMA (NVFP4: exact bf16 scaling); GEMM: 128-element chunks, compact fp32 table
// Decode is bound by the weight bytes in flight per SM: as many stages as shared memory holds
// next to the scale slices of a K = 5120 tile (1 byte per row and 64-block for NF4, 4 for the
// others; q8_0 stages are twice as large).
constexpr int decode_stages(int fmt) { return fmt == WQ_NF4 ? 6 : (fmt == WQ_Q8_0 || fmt == WQ_FP8) ? 3 : 4; }
constexpr int kGemmStagesP = 3;

template <int FMT>
int dispatch_p(const LinearArgs* probs, int count, bool out_f32, bool weights_static, cudaStream_t s) {
  int64_t maxM = 0;
  for (int i = 0; i < count; ++i) maxM = std::max(maxM, probs[i].M);
  int64_t maxK = 0;
  for (int i = 0; i < count; ++i) maxK = std::max(maxK, probs[i].K);
  if constexpr (Fmt<FMT>::UNIT) {
    // q4_1 / q5_0: encoder-sized GEMM tiles only (tcp_eligible keeps decode-sized problems off
    // this path); one 128-weight unit per chunk
    using Wide = PSmem<256, 2, FMT, 128, 1, kScaleF32>;
    if (maxK <= 64 * Wide::max_blocks())
      return launch_tcp<256, 2, FMT, 128, 1, kScaleF32>(probs, count, out_f32, weights_static, s);
    return launch_tcp<128, 2, FMT, 128, 1, kScaleF32>(probs, count, out_f32, weights_static, s);
  } else {
  // NVFP4 decodes E2M1 in registers (no table) and scales exactly in bf16
  if (maxM <= 16) {
    constexpr bool reg = FMT == WQ_NVFP4 || FMT == WQ_FP8;  // register decode, exact bf16 scaling
    constexpr int mode = reg ? kScaleBF16 : kScaleFold;
    constexpr int rep = reg ? 0 : 32;
    static_assert(PSmem<16, decode_stages(FMT), FMT, 256, rep, mode>::max_blocks() >= kMaxChunks,
                  "decode tiles must take K = 5120");
    return launch_tcp<16, decode_stages(FMT), FMT, 256, rep, mode>(probs, count, out_f32, weights_static, s);
  }
  // GEMM: 256 activation rows per tile (N = 256 MMAs, one TMEM accumulator) where shared memory
  // allows two stages of them and the scale slices of the longest K; else 128 rows (two accumulators)
  if constexpr (FMT == WQ_NVFP4 || FMT == WQ_FP8) {
    using Wide = PSmem<256, 2, FMT, 128, 0, kScaleBF16>;
    if (maxK <= 64 * Wide::max_blocks())
      return launch_tcp<256, 2, FMT, 128, 0, kScaleBF16>(probs, count, out_f32, weights_static, s);
    using Deep = PSmem<128, kGemmStagesP, FMT, 128, 0, kScaleBF16>;
    if (maxK <= 64 * Deep::max_blocks())
      return launch_tcp<128, kGemmStagesP, FMT, 128, 0, kScaleBF16>(probs, count, out_f32, weights_static, s);
    return launch_tcp<128, 2, FMT, 128, 0, kScaleBF16>(probs, count, out_f32, weights_static, s);
  }
  if constexpr (FMT == WQ_NF4) {
    using Wide = PSmem<256, 2, FMT, 128, 1, kScaleF32>;
    if (maxK <= 64 * Wide::max_blocks())
      return launch_tcp<256, 2, FMT, 128, 1, kScaleF32>(probs, count, out_f32, weights_static, s);
  }
  using Deep = PSmem<128, kGemmStagesP, FMT, 128, 1, kScaleF32>;
  if (maxK <= 64 * Deep::max_blocks())
    return launch_tcp<128, kGemmStagesP, FMT, 128, 1, kScaleF32>(probs, count, out_f32, weights_static, s);
  return launch_tcp<128, 2, FMT, 128, 1, kScaleF32>(probs, count, out_f32, weights_static, s);
  }
}

}  // namespace

bool tcp_eligible(const LinearArgs& a) {
  if (a.fmt != WQ_NF4 && a.fmt != WQ_NVFP4 && a.fmt != WQ_Q4_0 && a.fmt != WQ_Q8_0 && a.fmt != WQ_FP8 &&
      a.fmt != WQ_Q4_1 && a.fmt != WQ_Q5_0)
    return false;
  if ((a.fmt == WQ_Q4_1 || a.fmt == WQ_Q5_0) && a.M <= 16) return false;  // GEMM tiles only
  if (a.K % kKS != 0 || a.K < kKS || a.K > (int64_t)kKS * kMaxChunks) return false;
  if (a.M > 0x7FFFFFFF || a.N > 0x7FFFFFFF || a.K > 0x7FFFFFFF) return false;
  return ((uintptr_t)a.x & 15u) == 0;
}

int linear_tcp(const LinearArgs* probs, int count, cudaStream_t s) {
  if (count <= 0) return WQ_OK;
  const bool out_f32 = probs[0].out_f32, ws = probs[0].weights_static;
  switch (probs[0].fmt) {
    case WQ_NF4: return dispatch_p<WQ_NF4>(probs, count, out_f32, ws, s);
    case WQ_NVFP4: return dispatch_p<WQ_NVFP4>(probs, count, out_f32, ws, s);
    case WQ_Q4_0: return dispatch_p<WQ_Q4_0>(probs, count, out_f32, ws, s);
    case WQ_Q8_0: return dispatch_p<WQ_Q8_0>(probs, count, out_f32, ws, s);
    case WQ_FP8: return dispatch_p<WQ_FP8>(probs, count, out_f32, ws, s);
    case WQ_Q4_1: return dispatch_p<WQ_Q4_1>(probs, count, out_f32, ws, s);
    case WQ_Q5_0: return dispatch_p<WQ_Q5_0>(probs, count, out_f32, ws, s);
    default: return WQ_ERR_FMT;
  }
}

int take_status_tcp() {
  int v = 0, zero = 0;
  if (cudaMemcpyFromSymbol(&v, g_status, sizeof(int)) != cudaSuccess) return WQ_ERR_CUDA;
  cudaMemcpyToSymbol(g_status, &zero, sizeof(int));
  return v;
}

}  // namespace wq
