// wq_api.cu -- the C ABI of include/wq.h: argument checks, storage layout,
// dispatch between the tensor-core and CUDA-core paths.
#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <mutex>

#include "wq_internal.h"

namespace wq {

static std::atomic<uint64_t> g_launches{0};
void count_launch(int n) { g_launches.fetch_add((uint64_t)n, std::memory_order_relaxed); }

ScalesLayout scales_layout(int fmt, int64_t N, int64_t K) {
  ScalesLayout L;
  const int64_t n = N * K;
  switch (fmt) {
    case WQ_NF4: {
      const int64_t nb = n / 64;
      L.absmax_bytes = (size_t)nb;
      L.n_groups = (nb + 255) / 256;
      L.s2_off = align16((size_t)nb);
      L.offset_off = L.s2_off + 4 * (size_t)L.n_groups;
      L.total = L.offset_off + 4;
      break;
    }
    case WQ_NVFP4:
    case WQ_NVFP4_W4A4:
      L.sf_bytes = (size_t)(n / 16);
      L.g_off = align16(L.sf_bytes);
      L.total = L.g_off + 4;
      break;
    case WQ_Q4_0:
    case WQ_Q8_0:
    case WQ_Q5_0:
      L.total = align16((size_t)(n / 32) * 2);
      break;
    case WQ_Q4_1:
      L.total = 16;  // the (d, m) pairs live in the packed units; 16 zero bytes
      break;
    case WQ_FP8:
      L.total = align16((size_t)N * 4);
      break;
    default:
      break;
  }
  return L;
}

// cuTensorMapEncodeTiled through the runtime's driver entry point (no link-time libcuda dependency)
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn get_encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

bool encode_tmap_2d(void* tmap, CUtensorMapDataType dtype, const void* base, uint64_t inner, uint64_t outer,
                    uint64_t row_stride_bytes, uint32_t box_inner, uint32_t box_outer, CUtensorMapSwizzle swz) {
  EncodeTiledFn fn = get_encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {row_stride_bytes};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(reinterpret_cast<CUtensorMap*>(tmap), dtype, 2, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

int linear_one(const LinearArgs& a, cudaStream_t s) {
  int rc = WQ_OK;
  const bool dense = a.nout == 1 && a.ld[0] == a.N;
  if (a.fmt == WQ_NVFP4_W4A4) {
    if (dense && linear_w4a4_tc(a, s, &rc)) return rc;
  } else if (a.M <= 16) {
    // Measured on GB300 (back-to-back launches, NF4): one activation row runs fastest on the CUDA
    // cores (1280 x 1280: 3.5 us; 5120 x 1280: 5.0 us), as do up to 4 rows of a narrow or long-K
    // weight; the persistent tensor-core kernel (whole-K 128-row tiles) takes short-K Linears from
    // there on (5120 x 1280 at 4 rows: 6.1 against 9.9 us; 1280 x 1280 at 16 rows: 5.6 against
    // 8.3 us for the cluster split-K kernel, which keeps the long-K ones).
    const bool tcp_short = a.K <= kTcpDecodeMaxK && tcp_eligible(a);
    if (gemv_eligible(a) && (a.M == 1 || (a.M <= kGemvMaxM && !(tcp_short && a.N >= 4096))))
      return linear_gemv(a, s);
    if (tcp_short) return linear_tcp(&a, 1, s);
    if (dense && linear_tc(a, s, &rc)) return rc;
    if (gemv_eligible(a)) return linear_gemv(a, s);
  }
  if (a.fmt != WQ_NVFP4_W4A4 && dense && linear_w4a16_tc(a, s, &rc)) return rc;
  if (a.fmt != WQ_NVFP4_W4A4 && tcp_eligible(a)) return linear_tcp(&a, 1, s);
  return linear_simt(a, s);
}

}  // namespace wq

using namespace wq;

namespace {

inline bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

int block_of(int fmt) {
  switch (fmt) {
    case WQ_NF4: return 64;
    case WQ_NVFP4:
    case WQ_NVFP4_W4A4: return 32;  // 16-blocks; rows of packed codes must stay 16-byte aligned
    case WQ_Q4_0:
    case WQ_Q8_0:
    case WQ_FP8: return 32;
    case WQ_Q4_1:
    case WQ_Q5_0: return 128;  // whole 128-element storage units per row
    default: return 0;
  }
}

int check_weight(int fmt, int64_t N, int64_t K) {
  if (block_of(fmt) == 0) return WQ_ERR_FMT;
  if (N < 0 || K < 0) return WQ_ERR_ARG;
  if (K % block_of(fmt) != 0) return WQ_ERR_SHAPE;
  if (N > (int64_t(1) << 31) || K > (int64_t(1) << 31) || N * K > (int64_t(1) << 40)) return WQ_ERR_SHAPE;
  return WQ_OK;
}

int pack_common(int fmt, const float* W, int64_t N, int64_t K, void* packed, void* scales, void* stream,
                int (*fn)(const float*, int64_t, int64_t, uint8_t*, uint8_t*, cudaStream_t)) {
  int rc = check_weight(fmt, N, K);
  if (rc != WQ_OK) return rc;
  if (N * K == 0) return WQ_OK;
  if (!W || !packed || !scales) return WQ_ERR_ARG;
  if (!aligned16(W) || !aligned16(packed) || !aligned16(scales)) return WQ_ERR_ALIGN;
  return fn(W, N, K, reinterpret_cast<uint8_t*>(packed), reinterpret_cast<uint8_t*>(scales),
            reinterpret_cast<cudaStream_t>(stream));
}

}  // namespace

extern "C" {

size_t wq_packed_bytes(int fmt, int64_t N, int64_t K) {
  if (check_weight(fmt, N, K) != WQ_OK) return 0;
  return (size_t)(N * packed_row_bytes(fmt, K));
}

size_t wq_scales_bytes(int fmt, int64_t N, int64_t K) {
  if (check_weight(fmt, N, K) != WQ_OK) return 0;
  return scales_layout(fmt, N, K).total;
}

int wq_pack_nf4(const float* W, int64_t N, int64_t K, void* packed, void* scales, void* stream) {
  return pack_common(WQ_NF4, W, N, K, packed, scales, stream, pack_nf4);
}
int wq_pack_nvfp4(const float* W, int64_t N, int64_t K, void* packed, void* scales, void* stream) {
  return pack_common(WQ_NVFP4, W, N, K, packed, scales, stream, pack_nvfp4);
}
int wq_pack_q4_0(const float* W, int64_t N, int64_t K, void* packed, void* scales, void* stream) {
  return pack_common(WQ_Q4_0, W, N, K, packed, scales, stream, pack_q4_0);
}
int wq_pack_q8_0(const float* W, int64_t N, int64_t K, void* packed, void* scales, void* stream) {
  return pack_common(WQ_Q8_0, W, N, K, packed, scales, stream, pack_q8_0);
}

int wq_pack_q4_1(const float* W, int64_t N, int64_t K, void* packed, void* scales, void* stream) {
  return pack_common(WQ_Q4_1, W, N, K, packed, scales, stream, pack_q4_1);
}
int wq_pack_q5_0(const float* W, int64_t N, int64_t K, void* packed, void* scales, void* stream) {
  return pack_common(WQ_Q5_0, W, N, K, packed, scales, stream, pack_q5_0);
}
int wq_pack_fp8(const float* W, int64_t N, int64_t K, void* packed, void* scales, void* stream) {
  return pack_common(WQ_FP8, W, N, K, packed, scales, stream, pack_fp8);
}

int wq_dequant(const void* packed, const void* scales, int fmt, int64_t N, int64_t K, float* W_out, void* stream) {
  int rc = check_weight(fmt, N, K);
  if (rc != WQ_OK) return rc;
  if (N * K == 0) return WQ_OK;
  if (!packed || !scales || !W_out) return WQ_ERR_ARG;
  if (!aligned16(packed) || !aligned16(scales) || !aligned16(W_out)) return WQ_ERR_ALIGN;
  return dequant(reinterpret_cast<const uint8_t*>(packed), reinterpret_cast<const uint8_t*>(scales), fmt, N, K,
                 W_out, reinterpret_cast<cudaStream_t>(stream));
}

int wq_quant_act_nvfp4(const uint16_t* x, int64_t M, int64_t K, const float* g_in, uint8_t* codes, uint8_t* scales,
                       float* g_out, void* stream) {
  if (M < 0 || K < 0) return WQ_ERR_ARG;
  if (K % 32 != 0) return WQ_ERR_SHAPE;
  if (M * K == 0) return WQ_OK;
  if (!x || !codes || !scales || !g_out) return WQ_ERR_ARG;
  if (!aligned16(x) || !aligned16(codes) || !aligned16(scales) || ((uintptr_t)g_out & 3u) ||
      (g_in && ((uintptr_t)g_in & 3u)))
    return WQ_ERR_ALIGN;
  return quant_act_nvfp4(x, M, K, g_in, codes, scales, g_out, reinterpret_cast<cudaStream_t>(stream));
}

int wq_linear_ex(const void* x, const void* packed, const void* scales, int fmt, int64_t M, int64_t N, int64_t K,
                 const uint16_t* bias, void* y, unsigned flags, void* stream) {
  if (flags & ~(unsigned)(WQ_FLAG_OUT_F32 | WQ_FLAG_WEIGHTS_STATIC | WQ_FLAG_FORCE_SIMT)) return WQ_ERR_ARG;
  int rc = check_weight(fmt, N, K);
  if (rc != WQ_OK) return rc;
  if (M < 0) return WQ_ERR_ARG;
  if (M == 0 || N == 0) return WQ_OK;
  if (!x || !packed || !scales || !y) return WQ_ERR_ARG;
  if (!aligned16(packed) || !aligned16(scales) || !aligned16(y) || (bias && !aligned16(bias)))
    return WQ_ERR_ALIGN;
  LinearArgs a{};
  if (fmt == WQ_NVFP4_W4A4) {
    const wq_act_nvfp4* act = reinterpret_cast<const wq_act_nvfp4*>(x);  // host struct of device pointers
    if (!act->codes || !act->scales || !act->g) return WQ_ERR_ARG;
    if (!aligned16(act->codes) || !aligned16(act->scales) || ((uintptr_t)act->g & 3u)) return WQ_ERR_ALIGN;
    a.act_codes = act->codes;
    a.act_scales = act->scales;
    a.act_g = act->g;
  } else {
    if (!aligned16(x)) return WQ_ERR_ALIGN;
    a.x = x;
  }
  a.packed = reinterpret_cast<const uint8_t*>(packed);
  a.scales = reinterpret_cast<const uint8_t*>(scales);
  a.fmt = fmt;
  a.M = M;
  a.N = N;
  a.K = K;
  a.bias = bias;
  a.y = y;
  set_single_out(a);
  a.out_f32 = (flags & WQ_FLAG_OUT_F32) != 0;
  a.weights_static = (flags & WQ_FLAG_WEIGHTS_STATIC) != 0;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (flags & WQ_FLAG_FORCE_SIMT) return linear_simt(a, s);
  return linear_one(a, s);
}

int wq_linear_grouped(const wq_problem* problems, int count, int fmt, unsigned flags, void* stream) {
  if (!problems || count < 1 || count > WQ_GROUP_MAX) return WQ_ERR_ARG;
  wq_problem_ex ex[WQ_GROUP_MAX];
  for (int i = 0; i < count; ++i) {
    const wq_problem& p = problems[i];
    ex[i] = wq_problem_ex{};
    ex[i].x = p.x;
    ex[i].packed = p.packed;
    ex[i].scales = p.scales;
    ex[i].bias = p.bias;
    ex[i].M = p.M;
    ex[i].N = p.N;
    ex[i].K = p.K;
    ex[i].nout = 1;
    ex[i].out[0] = wq_out{p.y, p.N, p.N};
  }
  return wq_linear_grouped_ex(ex, count, fmt, flags, stream);
}

int wq_linear_grouped_ex(const wq_problem_ex* problems, int count, int fmt, unsigned flags, void* stream) {
  if (!problems || count < 1 || count > WQ_GROUP_MAX) return WQ_ERR_ARG;
  if (flags & ~(unsigned)(WQ_FLAG_OUT_F32 | WQ_FLAG_WEIGHTS_STATIC)) return WQ_ERR_ARG;
  if (fmt == WQ_NVFP4_W4A4) return WQ_ERR_FMT;
  const size_t esz = (flags & WQ_FLAG_OUT_F32) ? 4 : 2;
  LinearArgs args[WQ_GROUP_MAX];
  int n = 0;
  bool all_tc = true;
  for (int i = 0; i < count; ++i) {
    const wq_problem_ex& p = problems[i];
    int rc = check_weight(fmt, p.N, p.K);
    if (rc != WQ_OK) return rc;
    if (p.M < 0) return WQ_ERR_ARG;
    if (p.nout < 1 || p.nout > WQ_OUT_MAX) return WQ_ERR_ARG;
    if (p.M == 0 || p.N == 0) continue;
    if (!p.x || !p.packed || !p.scales) return WQ_ERR_ARG;
    if (!aligned16(p.x) || !aligned16(p.packed) || !aligned16(p.scales) || (p.bias && !aligned16(p.bias)))
      return WQ_ERR_ALIGN;
    LinearArgs a{};
    int64_t c = 0;
    for (int d = 0; d < p.nout; ++d) {
      const wq_out& o = p.out[d];
      if (!o.y || o.ncols <= 0 || o.ld < o.ncols) return WQ_ERR_ARG;
      if (d + 1 < p.nout && o.ncols % 16 != 0) return WQ_ERR_ARG;
      if (!aligned16(o.y) || ((size_t)o.ld * esz) % 16 != 0) return WQ_ERR_ALIGN;
      if (o.ld > 0x7FFFFFFF) return WQ_ERR_SHAPE;
      c += o.ncols;
      a.ys[d] = o.y;
      a.ld[d] = o.ld;
      a.col_end[d] = c;
    }
    if (c != p.N) return WQ_ERR_ARG;
    a.nout = p.nout;
    for (int d = p.nout; d < WQ_OUT_MAX; ++d) { a.ys[d] = a.ys[p.nout - 1]; a.ld[d] = a.ld[p.nout - 1]; a.col_end[d] = c; }
    a.x = p.x;
    a.y = p.out[0].y;
    a.packed = reinterpret_cast<const uint8_t*>(p.packed);
    a.scales = reinterpret_cast<const uint8_t*>(p.scales);
    a.fmt = fmt;
    a.M = p.M;
    a.N = p.N;
    a.K = p.K;
    a.bias = p.bias;
    a.out_f32 = (flags & WQ_FLAG_OUT_F32) != 0;
    a.weights_static = (flags & WQ_FLAG_WEIGHTS_STATIC) != 0;
    all_tc = all_tc && tcp_eligible(a);
    args[n++] = a;
  }
  if (n == 0) return WQ_OK;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (all_tc) return linear_tcp(args, n, s);
  for (int i = 0; i < n; ++i) {  // some problem outside the tensor-core rules: one launch each
    const int rc = linear_one(args[i], s);
    if (rc != WQ_OK) return rc;
  }
  return WQ_OK;
}

int wq_linear(const void* x, const void* packed, const void* scales, int fmt, int64_t M, int64_t N, int64_t K,
              const uint16_t* bias, void* y, void* stream) {
  return wq_linear_ex(x, packed, scales, fmt, M, N, K, bias, y, 0u, stream);
}

int wq_selftest_timeout(uint32_t polls, void* stream) {
  if (polls < 1 || polls > (1u << 20)) return WQ_ERR_ARG;
  return wq::selftest_timeout(polls, reinterpret_cast<cudaStream_t>(stream));
}

int wq_selftest_encoders(const float* in, int64_t n, uint8_t* out, void* stream) {
  if (n < 0 || n > (int64_t(1) << 30)) return WQ_ERR_ARG;
  if (n == 0) return WQ_OK;
  if (!in || !out) return WQ_ERR_ARG;
  if (!aligned16(in) || !aligned16(out)) return WQ_ERR_ALIGN;
  return wq::selftest_encoders(in, n, out, reinterpret_cast<cudaStream_t>(stream));
}

int wq_last_device_status(void) {
  if (cudaDeviceSynchronize() != cudaSuccess) return WQ_ERR_CUDA;
  int worst = WQ_OK;
  const int parts[6] = {take_status_pack(), take_status_simt(), take_status_tc(), take_status_tcp(),
                        take_status_w4a4(), take_status_w4a16()};
  for (int v : parts)
    if (v != WQ_OK) worst = v;
  return worst;
}

const char* wq_status_string(int status) {
  switch (status) {
    case WQ_OK: return "ok";
    case WQ_ERR_ARG: return "invalid argument (null pointer, negative size or unknown flag)";
    case WQ_ERR_SHAPE: return "unsupported shape (K not a multiple of the format's block, or too large)";
    case WQ_ERR_ALIGN: return "device pointer not 16-byte aligned";
    case WQ_ERR_FMT: return "unknown or unsupported format for this entry point";
    case WQ_ERR_CUDA: return "CUDA launch or runtime error";
    case WQ_ERR_TIMEOUT: return "a kernel abandoned a bounded wait";
    default: return "unknown status";
  }
}

uint64_t wq_kernel_launches(void) { return g_launches.load(std::memory_order_relaxed); }

}  // extern "C"
