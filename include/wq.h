/*
 * wq.h -- C ABI of libwq: fused dequantise-and-multiply of a block-quantised
 * Linear layer on GB300 (sm_103a),
 *
 *     y[M, N] = x[M, K] . dequant(W)[N, K]^T  (+ bias[N]).
 *
 * Source of the operation
 *   - PR "asr: add a 4-bit nf4 option for the Whisper engine", summary and
 *     "Why NF4 and not the NVFP4 snapshot": the weights are stored in 4 bits,
 *     activations stay bf16, and the dequantisation is fused into the matmul
 *     instead of unpacking W to bf16 and calling an ordinary GEMM.
 *   - model card "whisper-large-v3-turbo -- NVFP4", "What is quantized" and
 *     "Honest summary": NVFP4 weights (E2M1, E4M3 scale per 16, FP32 global
 *     scale) run as W4A16, and on Blackwell as W4A4 with activations
 *     quantised per 16 values at runtime.
 *   - PR "Run quantized Whisper on the fused Metal decode path", "Summary":
 *     GGUF q8_0 / q4_0 blocks of 32 with an fp16 scale.
 *
 * Conventions (all entry points)
 *   - W is PyTorch-Linear shaped, W[N, K] row-major, K contiguous; every
 *     quantisation block runs along K.  x is [M, K] row-major, y is [M, N]
 *     row-major.  bf16 / fp16 values are passed as their 16-bit patterns.
 *   - Every pointer argument is a DEVICE pointer unless stated otherwise.  The
 *     caller allocates and owns every buffer; the library never allocates,
 *     frees or synchronises (except wq_last_device_status).
 *   - Every call is asynchronous on `stream` (a cudaStream_t, NULL = legacy
 *     default stream) and returns a wq_status.  Arguments are checked before
 *     any launch; a failed check launches nothing.  No C++ exception crosses
 *     the ABI.
 *   - Device pointers must be 16-byte aligned (WQ_ERR_ALIGN otherwise).
 *   - Calls that share output buffers race if they overlap on the GPU; order
 *     them on one stream.
 */
#ifndef WQ_H_
#define WQ_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum wq_fmt {
  WQ_NF4 = 1,        /* NF4 codes, block 64, absmax double-quantised (int8 per 256, fp32 scale) */
  WQ_NVFP4 = 2,      /* E2M1 codes, block 16, E4M3 block scale, fp32 global; bf16 activations   */
  WQ_NVFP4_W4A4 = 3, /* NVFP4 weights AND NVFP4 activations (see wq_act_nvfp4)                   */
  WQ_Q4_0 = 4,       /* 4-bit codes, block 32, fp16 d, value (q - 8) * d                        */
  WQ_Q8_0 = 5,       /* int8 codes, block 32, fp16 d, value q * d                               */
  WQ_Q4_1 = 6,       /* 4-bit codes, block 32, fp16 d and fp16 minimum m, value q * d + m       */
  WQ_Q5_0 = 7,       /* 5-bit codes, block 32, fp16 d, value (q - 16) * d                       */
  WQ_FP8 = 8         /* FP8 E4M3 codes, one fp32 scale s per weight row, value E4M3(q) * s      */
} wq_fmt;

typedef enum wq_status {
  WQ_OK = 0,
  WQ_ERR_ARG = -1,     /* NULL pointer, unknown flag, negative size                    */
  WQ_ERR_SHAPE = -2,   /* K not a multiple of the format's block (or other size rule) */
  WQ_ERR_ALIGN = -3,   /* a device pointer is not 16-byte aligned                     */
  WQ_ERR_FMT = -4,     /* unknown format, or a format the entry point does not take   */
  WQ_ERR_CUDA = -5,    /* a CUDA launch / driver call failed                           */
  WQ_ERR_TIMEOUT = -6  /* a kernel gave up on a bounded wait (see wq_last_device_status) */
} wq_status;

/* Activations of WQ_NVFP4_W4A4, as written by wq_quant_act_nvfp4.  The struct
 * itself lives in HOST memory; its members are device pointers:
 *   codes  [M, K/2] bytes, two E2M1 codes per byte, element 2j in the low nibble
 *   scales [M, K/16] E4M3 bytes, row-major
 *   g      one fp32: the per-tensor decode multiplier                             */
typedef struct wq_act_nvfp4 {
  const uint8_t* codes;
  const uint8_t* scales;
  const float* g;
} wq_act_nvfp4;

/* ---------------------------------------------------------------- sizes
 * Bytes of the two buffers a packed weight occupies (0 for an invalid
 * format / shape).  Storage layout:
 *   packed  NF4, NVFP4, q4_0, q4_1: N*K/2 bytes, two codes per byte, element
 *           2j of the row-major flattening in the low nibble of byte j.
 *           q8_0: N*K int8.  FP8: N*K E4M3 bytes.
 *           q5_0, q4_1: N*K*5/8 bytes in 80-byte units, one per 128
 *           consecutive elements of a row: 64 bytes of (low) nibbles, element 2j
 *           in the low nibble of byte j, then 16 bytes of side data -- q5_0: the
 *           fifth bits (bit j of byte i = element 8i + j); q4_1: the unit's four
 *           (fp16 d, fp16 m) pairs, one per 32-block.
 *   scales  NF4:   int8 absmax codes [N*K/64] | zero pad to 16 B |
 *                  fp32 second-level scale s2 [ceil(N*K/64 / 256)] | fp32 offset
 *           NVFP4: E4M3 block scales [N, K/16] row-major | zero pad to 16 B | fp32 g
 *           q4_0, q8_0, q5_0: fp16 d [N*K/32] | zero pad to 16 B
 *           q4_1:  16 zero bytes (its scales are inside the packed units)
 *           FP8:   fp32 s [N] | zero pad to 16 B
 * Size rules: NF4 K % 64 == 0; NVFP4 K % 32 == 0; q4_0 / q8_0 / FP8
 * K % 32 == 0; q5_0 / q4_1 K % 128 == 0.                                      */
size_t wq_packed_bytes(int fmt, int64_t N, int64_t K);
size_t wq_scales_bytes(int fmt, int64_t N, int64_t K);

/* ---------------------------------------------------------------- packers
 * Quantise fp32 weights W [N, K] (device) into `packed` and `scales` (device,
 * sizes above).  Deterministic and bit-identical for a given W.  The packers
 * use `packed` as working space before writing it, so W must not alias either
 * output.  WQ_NVFP4_W4A4 weights are packed with wq_pack_nvfp4.
 *
 * wq_pack_nf4   (PR "asr: add a 4-bit nf4 option ...", "What's here"):
 *   per 64-block absmax a; code = number of NF4 codebook midpoints below w / a
 *   (ties to the lower code); the absmax values are centred on their exact
 *   mean (fp32 offset) and quantised to int8 per group of 256 with an fp32
 *   scale s2 = max|a - offset| / 127.
 * wq_pack_nvfp4 (model card "whisper-large-v3-turbo -- NVFP4",
 *   "What is quantized"): g = amax(W) / 2688; per 16-block
 *   s = E4M3((amax_b / 6) / g), code = E2M1(w / (E4M3(s) * g)); round to
 *   nearest even, saturating.
 * wq_pack_q4_0  (PR "Run quantized Whisper on the fused Metal decode path",
 *   "Summary"): d = fp16(extreme / -8), q = clamp(rint(w / d) + 8, 0, 15).
 * wq_pack_q8_0  (same passage): d = fp16(amax / 127), q = clamp(rint(w / d), +-127).
 * wq_pack_q4_1, wq_pack_q5_0 (same PR, "Why the policy": the other GGUF block
 *   types): q4_1 m = fp16(min), d = fp16((max - min) / 15),
 *   q = clamp(rint((w - m) / d), 0, 15); q5_0 d = fp16(extreme / -16),
 *   q = clamp(rint(w / d) + 16, 0, 31).
 * wq_pack_fp8   (model card "whisper-large-v3-turbo -- NVFP4", "Honest
 *   summary": the FP8 build): s = amax(row) / 448, q = E4M3(w / s), round to
 *   nearest even, saturating (q = 0 for an all-zero row).
 * Every rint / E4M3 rounding is half to even, against the stored fp16 / fp32
 * scale values.
 */
int wq_pack_nf4(const float* W, int64_t N, int64_t K, void* packed, void* scales, void* stream);
int wq_pack_nvfp4(const float* W, int64_t N, int64_t K, void* packed, void* scales, void* stream);
int wq_pack_q4_0(const float* W, int64_t N, int64_t K, void* packed, void* scales, void* stream);
int wq_pack_q8_0(const float* W, int64_t N, int64_t K, void* packed, void* scales, void* stream);
int wq_pack_q4_1(const float* W, int64_t N, int64_t K, void* packed, void* scales, void* stream);
int wq_pack_q5_0(const float* W, int64_t N, int64_t K, void* packed, void* scales, void* stream);
int wq_pack_fp8(const float* W, int64_t N, int64_t K, void* packed, void* scales, void* stream);

/* ---------------------------------------------------------------- dequant
 * Decode a packed weight to fp32 W_out [N, K] (device): the exact fp32 value
 * each code stands for (NF4: codebook * (q*s2 + offset); NVFP4:
 * (E2M1 * E4M3) * g; q4_0: (q-8)*d; q8_0: q*d; q4_1: q*d + m; q5_0:
 * (q-16)*d; FP8: E4M3(q)*s).  A verification export: the
 * fused paths below never materialise W.                                       */
int wq_dequant(const void* packed, const void* scales, int fmt, int64_t N, int64_t K,
               float* W_out, void* stream);

/* ---------------------------------------------------------------- activations
 * NVFP4 runtime activation quantiser (model card "whisper-large-v3-turbo --
 * NVFP4", "What is quantized": activations quantised per 16-value group at
 * runtime).  x: bf16 [M, K] (K % 32 == 0).  g_in: NULL for a dynamic
 * per-tensor global g = amax(x) / 2688 (1 if x is all zero), or a device
 * pointer to a static fp32 g.  Writes codes [M, K/2], scales [M, K/16] and
 * g_out (one fp32, the g that was used).  Bit-identical to the block encoder
 * of wq_pack_nvfp4.                                                            */
int wq_quant_act_nvfp4(const uint16_t* x, int64_t M, int64_t K, const float* g_in,
                       uint8_t* codes, uint8_t* scales, float* g_out, void* stream);

/* ---------------------------------------------------------------- linear
 * y = x . dequant(W)^T (+ bias), fp32 accumulation, bf16 output.
 *   x      bf16 [M, K]; for WQ_NVFP4_W4A4 a HOST pointer to a wq_act_nvfp4
 *   bias   bf16 [N] or NULL
 *   y      bf16 [M, N]
 * M == 0 is a no-op.  Dispatch: M <= 16 runs the decode path (tensor-core
 * GEMV, split-K over a thread-block cluster); larger M runs the persistent
 * tensor-core GEMM; K not a multiple of 64 runs a CUDA-core kernel with the
 * same per-weight decode.  WQ_NVFP4_W4A4 with M > 16 and K a multiple of 256
 * runs the block-scaled FP4 tensor-core GEMM (both operands packed); other
 * W4A4 shapes run the CUDA-core kernel.                                         */
int wq_linear(const void* x, const void* packed, const void* scales, int fmt,
              int64_t M, int64_t N, int64_t K, const uint16_t* bias, void* y, void* stream);

/* Flags of wq_linear_ex. */
enum {
  /* y is fp32 [M, N] instead of bf16 (same kernels; the final bf16 rounding is skipped). */
  WQ_FLAG_OUT_F32 = 1u << 0,
  /* The caller promises that `packed`, `scales` and `bias` are not written by
   * work still running on `stream`.  The kernel is then launched with
   * programmatic dependent launch and starts streaming its weights before the
   * preceding kernel on the stream has finished; it waits for that kernel
   * only before it reads x or writes y.                                        */
  WQ_FLAG_WEIGHTS_STATIC = 1u << 1,
  /* Force the CUDA-core path (verification aid). */
  WQ_FLAG_FORCE_SIMT = 1u << 2
};

int wq_linear_ex(const void* x, const void* packed, const void* scales, int fmt,
                 int64_t M, int64_t N, int64_t K, const uint16_t* bias, void* y,
                 unsigned flags, void* stream);

/* ---------------------------------------------------------------- grouped
 * Several independent Linears of ONE format in one launch (the fused Q/K/V
 * projection of PR "Run quantized Whisper on the fused Metal decode path",
 * "Summary", generalised to any set of Linears whose inputs are ready).  Each
 * problem has the meaning of one wq_linear call (same layouts and rules);
 * outputs must not overlap.  `problems` is a HOST array of `count` entries,
 * 1 <= count <= WQ_GROUP_MAX; WQ_NVFP4_W4A4 is not accepted (WQ_ERR_FMT).
 * flags: WQ_FLAG_OUT_F32 / WQ_FLAG_WEIGHTS_STATIC apply to every problem.     */
#define WQ_GROUP_MAX 48
typedef struct wq_problem {
  const void* x;          /* bf16 [M, K]          */
  const void* packed;     /* packed weight        */
  const void* scales;     /* its scales blob      */
  const uint16_t* bias;   /* bf16 [N] or NULL     */
  void* y;                /* bf16 (or fp32) [M, N] */
  int64_t M, N, K;
} wq_problem;

int wq_linear_grouped(const wq_problem* problems, int count, int fmt, unsigned flags, void* stream);

/* ---------------------------------------------------------------- grouped, strided outputs
 * wq_linear_grouped_ex: as wq_linear_grouped, but each problem's output columns
 * go to up to WQ_OUT_MAX row-strided destinations instead of one dense y.  This
 * is the fused Q/K/V projection of PR "Run quantized Whisper on the fused Metal
 * decode path", "Summary" and "Test plan": the projections of a token are
 * computed in one launch, the bias added on the device, and K and V written
 * straight into their rows of a KV-cache slab, with no copy afterwards.  It
 * also serves a merged weight: the cross-attention K and V weights stacked as
 * one [2N, K] matrix (packed once), whose first N output columns go to the K
 * slab and the last N to the V slab.
 *
 * Destination d of a problem receives the output columns
 * [c_d, c_d + out[d].ncols), c_d = out[0].ncols + ... + out[d-1].ncols: element
 * (m, n) is written to out[d].y + m * out[d].ld + (n - c_d) (elements of bf16, or
 * fp32 with WQ_FLAG_OUT_F32).  Rules (WQ_ERR_ARG / WQ_ERR_ALIGN otherwise):
 * 1 <= nout <= WQ_OUT_MAX; the ncols sum to N; every ncols but the last is a
 * multiple of 16; ld >= ncols and ld * element size is a multiple of 16 bytes;
 * every y is 16-byte aligned.  Destinations must not overlap each other or any
 * other problem's.  Nothing outside the addressed elements is written: rows of
 * a slab other than the M addressed ones, and the columns of a row beyond
 * ncols, keep their contents.                                                  */
#define WQ_OUT_MAX 4
typedef struct wq_out {
  void* y;         /* first element of the destination (device)   */
  int64_t ld;      /* row stride in elements                       */
  int64_t ncols;   /* output columns this destination receives     */
} wq_out;

typedef struct wq_problem_ex {
  const void* x;          /* bf16 [M, K]                              */
  const void* packed;     /* packed weight [N, K]                     */
  const void* scales;     /* its scales blob                          */
  const uint16_t* bias;   /* bf16 [N] or NULL                         */
  int64_t M, N, K;
  int nout;               /* destinations used, 1 .. WQ_OUT_MAX        */
  wq_out out[WQ_OUT_MAX];
} wq_problem_ex;

int wq_linear_grouped_ex(const wq_problem_ex* problems, int count, int fmt, unsigned flags, void* stream);

/* ---------------------------------------------------------------- status
 * wq_last_device_status: synchronises the current device, returns and clears
 * the device-side status word (WQ_OK, or WQ_ERR_TIMEOUT if a kernel abandoned
 * a bounded wait since the last call).  Not for hot loops.
 * wq_status_string: a static description of a status code.
 * wq_kernel_launches: number of kernels this library has launched in this
 * process (host-side counter).                                                 */
int wq_last_device_status(void);
const char* wq_status_string(int status);
uint64_t wq_kernel_launches(void);

/* ---------------------------------------------------------------- failure detection
 * wq_selftest_timeout: launches one small kernel that waits, with the same
 * bounded mbarrier poll every kernel of this library uses, on a barrier that
 * nothing ever arrives on, giving up after `polls` polls (1 <= polls <= 2^20).
 * The kernel then records WQ_ERR_TIMEOUT in the device status word and
 * returns normally: no trap, the context stays usable.  A following
 * wq_last_device_status() returns WQ_ERR_TIMEOUT (and clears it).  Exercises
 * the path a real stall takes (a TMA transaction or a peer that never
 * arrives) without faulting the GPU.  WQ_ERR_ARG for polls out of range.    */
int wq_selftest_timeout(uint32_t polls, void* stream);

/* ---------------------------------------------------------------- encoder check
 * wq_selftest_encoders: a verification export.  For each of the n fp32 values
 * in[i] (device), writes four bytes out[4i .. 4i+3] (device):
 *   [0] the E2M1 code the library's packers / activation quantiser assign
 *   [1] the E2M1 code of the hardware conversion cvt.rn.satfinite.e2m1x2.f32
 *   [2] the E4M3 byte the library's block-scale encoder assigns
 *   [3] the E4M3 byte of cvt.rn.satfinite.e4m3x2.f32
 * so that tests can pin both the library's encoders (model card
 * "whisper-large-v3-turbo -- NVFP4", "What is quantized": E2M1 codes, E4M3
 * block scales) and the hardware's rounding of ties and signed zeros.
 * WQ_ERR_ARG for n < 0 or n > 2^30, WQ_ERR_ALIGN for unaligned pointers.     */
int wq_selftest_encoders(const float* in, int64_t n, uint8_t* out, void* stream);

#ifdef __cplusplus
}
#endif
#endif /* WQ_H_ */
