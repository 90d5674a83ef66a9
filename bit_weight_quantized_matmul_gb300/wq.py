"""ctypes binding of libwq (include/wq.h): argument marshalling only.

Every compute step runs in libwq's CUDA kernels.  Importing this module loads
``libwq.so`` from this package directory and raises ImportError when it is
missing (build it with ``python -m bit_weight_quantized_matmul_gb300.build``);
there is no fallback implementation.  The C entry points keep their names
(``wq_linear`` ...); the torch helpers below allocate outputs with torch and
pass raw device pointers plus the current CUDA stream.
"""
import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libwq.so")

if not os.path.exists(LIB_PATH):
    raise ImportError(f"libwq.so not found at {LIB_PATH}: build it first "
                      f"(python -m bit_weight_quantized_matmul_gb300.build)")
lib = ctypes.CDLL(LIB_PATH)

# ------------------------------------------------------------------ constants
WQ_NF4, WQ_NVFP4, WQ_NVFP4_W4A4, WQ_Q4_0, WQ_Q8_0, WQ_Q4_1, WQ_Q5_0, WQ_FP8 = 1, 2, 3, 4, 5, 6, 7, 8
FMT = {"nf4": WQ_NF4, "nvfp4": WQ_NVFP4, "nvfp4_w4a4": WQ_NVFP4_W4A4, "q4_0": WQ_Q4_0, "q8_0": WQ_Q8_0,
       "q4_1": WQ_Q4_1, "q5_0": WQ_Q5_0, "fp8": WQ_FP8}
WQ_OK, WQ_ERR_ARG, WQ_ERR_SHAPE, WQ_ERR_ALIGN, WQ_ERR_FMT, WQ_ERR_CUDA, WQ_ERR_TIMEOUT = 0, -1, -2, -3, -4, -5, -6
WQ_FLAG_OUT_F32, WQ_FLAG_WEIGHTS_STATIC, WQ_FLAG_FORCE_SIMT = 1, 2, 4


class wq_act_nvfp4(ctypes.Structure):
    _fields_ = [("codes", ctypes.c_void_p), ("scales", ctypes.c_void_p), ("g", ctypes.c_void_p)]


class wq_problem(ctypes.Structure):
    _fields_ = [("x", ctypes.c_void_p), ("packed", ctypes.c_void_p), ("scales", ctypes.c_void_p),
                ("bias", ctypes.c_void_p), ("y", ctypes.c_void_p), ("M", ctypes.c_int64),
                ("N", ctypes.c_int64), ("K", ctypes.c_int64)]


WQ_GROUP_MAX = 48
WQ_OUT_MAX = 4


class wq_out(ctypes.Structure):
    _fields_ = [("y", ctypes.c_void_p), ("ld", ctypes.c_int64), ("ncols", ctypes.c_int64)]


class wq_problem_ex(ctypes.Structure):
    _fields_ = [("x", ctypes.c_void_p), ("packed", ctypes.c_void_p), ("scales", ctypes.c_void_p),
                ("bias", ctypes.c_void_p), ("M", ctypes.c_int64), ("N", ctypes.c_int64), ("K", ctypes.c_int64),
                ("nout", ctypes.c_int), ("out", wq_out * WQ_OUT_MAX)]

_P, _I64, _I, _U = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_uint
_SIGS = {
    "wq_packed_bytes": (ctypes.c_size_t, [_I, _I64, _I64]),
    "wq_scales_bytes": (ctypes.c_size_t, [_I, _I64, _I64]),
    "wq_pack_nf4": (_I, [_P, _I64, _I64, _P, _P, _P]),
    "wq_pack_nvfp4": (_I, [_P, _I64, _I64, _P, _P, _P]),
    "wq_pack_q4_0": (_I, [_P, _I64, _I64, _P, _P, _P]),
    "wq_pack_q8_0": (_I, [_P, _I64, _I64, _P, _P, _P]),
    "wq_pack_q4_1": (_I, [_P, _I64, _I64, _P, _P, _P]),
    "wq_pack_q5_0": (_I, [_P, _I64, _I64, _P, _P, _P]),
    "wq_pack_fp8": (_I, [_P, _I64, _I64, _P, _P, _P]),
    "wq_dequant": (_I, [_P, _P, _I, _I64, _I64, _P, _P]),
    "wq_quant_act_nvfp4": (_I, [_P, _I64, _I64, _P, _P, _P, _P, _P]),
    "wq_linear": (_I, [_P, _P, _P, _I, _I64, _I64, _I64, _P, _P, _P]),
    "wq_linear_ex": (_I, [_P, _P, _P, _I, _I64, _I64, _I64, _P, _P, _U, _P]),
    "wq_linear_grouped": (_I, [_P, _I, _I, _U, _P]),
    "wq_linear_grouped_ex": (_I, [_P, _I, _I, _U, _P]),
    "wq_last_device_status": (_I, []),
    "wq_status_string": (ctypes.c_char_p, [_I]),
    "wq_kernel_launches": (ctypes.c_uint64, []),
    "wq_selftest_timeout": (_I, [ctypes.c_uint32, _P]),
    "wq_selftest_encoders": (_I, [_P, _I64, _P, _P]),
}
for _name, (_res, _args) in _SIGS.items():
    _f = getattr(lib, _name)
    _f.restype = _res
    _f.argtypes = _args
    globals()[_name] = _f


class WQError(RuntimeError):
    def __init__(self, where, status):
        super().__init__(f"{where}: {lib.wq_status_string(status).decode()} (status {status})")
        self.status = status


def _check(where, status):
    if status != WQ_OK:
        raise WQError(where, status)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _fmt(fmt):
    return FMT[fmt] if isinstance(fmt, str) else int(fmt)


# ------------------------------------------------------------------ torch helpers
def packed_bytes(fmt, N, K):
    return int(lib.wq_packed_bytes(_fmt(fmt), N, K))


def scales_bytes(fmt, N, K):
    return int(lib.wq_scales_bytes(_fmt(fmt), N, K))


def alloc_packed(fmt, N, K, device="cuda"):
    pb, sb = packed_bytes(fmt, N, K), scales_bytes(fmt, N, K)
    if pb == 0 and N * K != 0:
        raise WQError("alloc_packed", WQ_ERR_SHAPE)
    return (torch.empty(max(pb, 16), dtype=torch.uint8, device=device),
            torch.empty(max(sb, 16), dtype=torch.uint8, device=device))


_PACK_FN = {"nf4": "wq_pack_nf4", "nvfp4": "wq_pack_nvfp4", "nvfp4_w4a4": "wq_pack_nvfp4",
            "q4_0": "wq_pack_q4_0", "q8_0": "wq_pack_q8_0", "q4_1": "wq_pack_q4_1", "q5_0": "wq_pack_q5_0",
            "fp8": "wq_pack_fp8"}


def pack(fmt, W, out=None, stream=None):
    """Quantise fp32 W [N, K] (CUDA) -> (packed, scales) uint8 CUDA tensors."""
    assert W.is_cuda and W.dtype == torch.float32 and W.is_contiguous()
    N, K = W.shape
    packed, scales = alloc_packed(fmt, N, K, W.device) if out is None else out
    _check(_PACK_FN[fmt], getattr(lib, _PACK_FN[fmt])(_ptr(W), N, K, _ptr(packed), _ptr(scales), _stream(stream)))
    return packed, scales


def dequant(fmt, packed, scales, N, K, stream=None):
    out = torch.empty((N, K), dtype=torch.float32, device=packed.device)
    _check("wq_dequant", lib.wq_dequant(_ptr(packed), _ptr(scales), _fmt(fmt), N, K, _ptr(out), _stream(stream)))
    return out


def quant_act_nvfp4(x, g_in=None, out=None, stream=None):
    """x bf16 [M, K] (CUDA) -> (codes [M, K/2], scales [M, K/16], g [1]) CUDA tensors."""
    assert x.is_cuda and x.dtype == torch.bfloat16 and x.is_contiguous()
    M, K = x.shape
    if out is None:
        codes = torch.empty((M, K // 2), dtype=torch.uint8, device=x.device)
        scales = torch.empty((M, K // 16), dtype=torch.uint8, device=x.device)
        g = torch.empty(1, dtype=torch.float32, device=x.device)
    else:
        codes, scales, g = out
    _check("wq_quant_act_nvfp4", lib.wq_quant_act_nvfp4(_ptr(x), M, K, _ptr(g_in), _ptr(codes), _ptr(scales),
                                                        _ptr(g), _stream(stream)))
    return codes, scales, g


def act_struct(codes, scales, g):
    return wq_act_nvfp4(codes.data_ptr(), scales.data_ptr(), g.data_ptr())


def linear_into(y, x, packed, scales, fmt, N, K, bias=None, out_f32=False, weights_static=False,
                force_simt=False, stream=None):
    """y = x . dequant(W)^T (+ bias) into a preallocated y.  For fmt 'nvfp4_w4a4', x is the
    (codes, scales, g) triple of quant_act_nvfp4."""
    f = _fmt(fmt)
    flags = (WQ_FLAG_OUT_F32 if out_f32 else 0) | (WQ_FLAG_WEIGHTS_STATIC if weights_static else 0) | \
        (WQ_FLAG_FORCE_SIMT if force_simt else 0)
    if f == WQ_NVFP4_W4A4:
        codes, sc, g = x
        M = codes.shape[0]
        act = act_struct(codes, sc, g)
        xp = ctypes.cast(ctypes.pointer(act), ctypes.c_void_p)
    else:
        M = x.shape[0]
        xp = _ptr(x)
    _check("wq_linear_ex", lib.wq_linear_ex(xp, _ptr(packed), _ptr(scales), f, M, N, K, _ptr(bias), _ptr(y),
                                            flags, _stream(stream)))
    return y


def linear(x, packed, scales, fmt, N, K, bias=None, out_f32=False, weights_static=False, force_simt=False,
           stream=None):
    M = (x[0].shape[0] if _fmt(fmt) == WQ_NVFP4_W4A4 else x.shape[0])
    dev = x[0].device if _fmt(fmt) == WQ_NVFP4_W4A4 else x.device
    y = torch.empty((M, N), dtype=torch.float32 if out_f32 else torch.bfloat16, device=dev)
    return linear_into(y, x, packed, scales, fmt, N, K, bias, out_f32, weights_static, force_simt, stream)


def linear_grouped(problems, fmt, out_f32=False, weights_static=False, stream=None):
    """Independent Linears of one format in one launch.  ``problems`` is a list of
    (y, x, packed, scales, N, K, bias) tuples; each y [M, N] is written in place."""
    arr = (wq_problem * len(problems))()
    for i, (y, x, packed, scales, N, K, bias) in enumerate(problems):
        arr[i] = wq_problem(x.data_ptr(), packed.data_ptr(), scales.data_ptr(),
                            None if bias is None else bias.data_ptr(), y.data_ptr(), x.shape[0], N, K)
    flags = (WQ_FLAG_OUT_F32 if out_f32 else 0) | (WQ_FLAG_WEIGHTS_STATIC if weights_static else 0)
    _check("wq_linear_grouped", lib.wq_linear_grouped(ctypes.cast(arr, ctypes.c_void_p), len(problems),
                                                      _fmt(fmt), flags, _stream(stream)))


def linear_grouped_ex(problems, fmt, out_f32=False, weights_static=False, stream=None):
    """Independent Linears of one format in one launch, each writing its output columns to up to
    WQ_OUT_MAX row-strided destinations.  ``problems`` is a list of (x, packed, scales, N, K, bias,
    outs) with ``outs`` a list of (view, ncols): ``view`` is a 2-D CUDA tensor view whose first M rows
    (row stride ``view.stride(0)``) receive the next ``ncols`` output columns."""
    arr = (wq_problem_ex * len(problems))()
    for i, (x, packed, scales, N, K, bias, outs) in enumerate(problems):
        pe = wq_problem_ex()
        pe.x, pe.packed, pe.scales = x.data_ptr(), packed.data_ptr(), scales.data_ptr()
        pe.bias = None if bias is None else bias.data_ptr()
        pe.M, pe.N, pe.K, pe.nout = x.shape[0], N, K, len(outs)
        for d, (view, ncols) in enumerate(outs):
            pe.out[d] = wq_out(view.data_ptr(), view.stride(0), ncols)
        arr[i] = pe
    flags = (WQ_FLAG_OUT_F32 if out_f32 else 0) | (WQ_FLAG_WEIGHTS_STATIC if weights_static else 0)
    _check("wq_linear_grouped_ex", lib.wq_linear_grouped_ex(ctypes.cast(arr, ctypes.c_void_p), len(problems),
                                                            _fmt(fmt), flags, _stream(stream)))


def last_device_status():
    return int(lib.wq_last_device_status())


def kernel_launches():
    return int(lib.wq_kernel_launches())


def selftest_timeout(polls=1000, stream=None):
    """Run the bounded-wait failure path once (a barrier nobody arrives on); the next
    last_device_status() reports WQ_ERR_TIMEOUT."""
    _check("wq_selftest_timeout", lib.wq_selftest_timeout(polls, _stream(stream)))


def selftest_encoders(x, stream=None):
    """fp32 CUDA tensor x -> uint8 [n, 4]: (library E2M1, hardware E2M1, library E4M3,
    hardware E4M3) codes of every value."""
    assert x.is_cuda and x.dtype == torch.float32 and x.is_contiguous()
    out = torch.empty((x.numel(), 4), dtype=torch.uint8, device=x.device)
    _check("wq_selftest_encoders", lib.wq_selftest_encoders(_ptr(x), x.numel(), _ptr(out), _stream(stream)))
    return out
