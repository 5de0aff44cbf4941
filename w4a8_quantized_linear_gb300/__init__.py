"""GB300-native W8A8 / W4A8 online-activation-quantized linear layer.

A thin binding over the C ABI of ``libcider.so`` (declared in
``include/cider.h``).  Each function here has the name of the C entry point it
calls, takes PyTorch CUDA tensors, allocates the outputs with PyTorch on the
input's device, and passes raw pointers and the current CUDA stream.  Every
step of the computation runs in the library's CUDA kernels; there is no CPU or
PyTorch fallback: if the library is missing or the GPU is not sm_103, calls
raise.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

from . import inputs  # noqa: F401  (seeded synthetic inputs, no arithmetic)

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "_build", "libcider.so")
HEADER_PATH = os.path.join(os.path.dirname(_PKG), "include", "cider.h")

CIDER_OK = 0
CIDER_PER_CHANNEL = 0
CIDER_PER_GROUP = 1
CIDER_F16 = 0
CIDER_BF16 = 1
_DTYPES = {torch.float16: CIDER_F16, torch.bfloat16: CIDER_BF16}
STATUS_NAMES = {0: "CIDER_OK", 1: "CIDER_ERR_INVALID_ARGUMENT", 2: "CIDER_ERR_MISALIGNED",
                3: "CIDER_ERR_UNSUPPORTED_DEVICE", 4: "CIDER_ERR_CUDA", 5: "CIDER_ERR_TIMEOUT"}

_lib = None
_lock = threading.Lock()


class CiderError(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        msg = _load().cider_status_string(status).decode()
        super().__init__(f"{fn} failed with status {status}: {msg}")


def _declare(lib):
    p, i64, i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
    sig = {
        "cider_is_available": ([], i32),
        "cider_status_string": ([i32], ctypes.c_char_p),
        "cider_version": ([], i32),
        "cider_quantize_act": ([p, i64, i64, p, p, p], i32),
        "cider_quantize_act_bf16": ([p, i64, i64, p, p, p], i32),
        "cider_int4_from_offset_binary": ([p, p, i64, p], i32),
        "cider_quantize_weight_int8": ([p, i64, i64, i32, p, p, p], i32),
        "cider_quantize_weight_int4": ([p, i64, i64, i32, p, p, p], i32),
        "cider_quantize_weight_int8_clip": ([p, i64, i64, i32, ctypes.c_double, p, p, p], i32),
        "cider_quantize_weight_int4_clip": ([p, i64, i64, i32, ctypes.c_double, p, p, p], i32),
        "cider_w8a8_linear": ([p, i64, i64, i64, p, p, i32, i32, p, p], i32),
        "cider_w4a8_linear": ([p, i64, i64, i64, p, p, i32, i32, p, p], i32),
        "cider_w8a8_linear_bf16": ([p, i64, i64, i64, p, p, i32, i32, p, p], i32),
        "cider_w4a8_linear_bf16": ([p, i64, i64, i64, p, p, i32, i32, p, p], i32),
        "cider_w8a8_linear_ex": ([p, i32, i64, i64, i64, p, p, i32, i32, p, i32, p], i32),
        "cider_w4a8_linear_ex": ([p, i32, i64, i64, i64, p, p, i32, i32, p, i32, p], i32),
        "cider_w8a8_linear_prequant": ([p, p, i64, i64, i64, p, p, i32, i32, p, p], i32),
        "cider_w4a8_linear_prequant": ([p, p, i64, i64, i64, p, p, i32, i32, p, p], i32),
        "cider_w8a8_accumulators": ([p, i64, i64, i64, p, i32, p, p], i32),
        "cider_w4a8_accumulators": ([p, i64, i64, i64, p, i32, p, p], i32),
        "cider_check_device_error": ([p], i32),
        "cider_trim_scratch_pool": ([i64, p], i32),
        "cider_timing_begin": ([i64], i32),
        "cider_timing_end": ([ctypes.POINTER(i64), ctypes.POINTER(ctypes.c_double)], i32),
        "cider_debug_wait_timeout": ([i64, p], i32),
        "cider_debug_pair_schedule": ([i64, i64, i64, i32, i64, p, p, p], i32),
        "cider_debug_small_m_slices": ([i64, i64, i64, i32, i32, i32, p], i32),
        "cider_debug_small_m_launch": ([i64, i64, i64, i32, i32, i32, i32, p], i32),
    }
    for name, (args, res) in sig.items():
        f = getattr(lib, name)
        f.argtypes = args
        f.restype = res
    return lib


def _load():
    """Load libcider.so (built in-tree by ``_build.build()``); raise if absent."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(
                    f"libcider.so not found at {LIB_PATH}: build it first with "
                    "`python -m w4a8_quantized_linear_gb300._build` (needs nvcc); "
                    "there is no fallback implementation")
            _lib = _declare(ctypes.CDLL(LIB_PATH))
    return _lib


def library():
    """The loaded ctypes library (for callers that want the raw C ABI)."""
    return _load()


def _check(fn: str, status: int):
    if status != CIDER_OK:
        raise CiderError(fn, status)


def _stream(t: torch.Tensor):
    return ctypes.c_void_p(torch.cuda.current_stream(t.device).cuda_stream)


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else None


def _need(t: torch.Tensor, dtype, name: str, ndim: int):
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dimensions, got shape {tuple(t.shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


# ----------------------------------------------------------------------------- API
def cider_is_available() -> bool:
    return bool(_load().cider_is_available())


def _quantize_act(fn, x, dtype):
    _need(x, dtype, "x", 2)
    M, K = x.shape
    qa = torch.empty((M, K), dtype=torch.int8, device=x.device)
    sa = torch.empty((M,), dtype=torch.float32, device=x.device)
    _check(fn, getattr(_load(), fn)(_ptr(x), M, K, _ptr(qa), _ptr(sa), _stream(x)))
    return qa, sa


def cider_quantize_act(x: torch.Tensor):
    """x fp16 [M, K] -> (qa int8 [M, K], sa fp32 [M])."""
    return _quantize_act("cider_quantize_act", x, torch.float16)


def cider_quantize_act_bf16(x: torch.Tensor):
    """x bf16 [M, K] -> (qa int8 [M, K], sa fp32 [M])."""
    return _quantize_act("cider_quantize_act_bf16", x, torch.bfloat16)


def cider_int4_from_offset_binary(packed: torch.Tensor, out=None):
    """uint8 INT4 bytes stored offset-binary (nibble u = value + 8) -> the
    library's two's complement packing (out may be packed itself)."""
    if not isinstance(packed, torch.Tensor) or not packed.is_cuda or packed.dtype != torch.uint8:
        raise TypeError("packed must be a CUDA uint8 tensor")
    if not packed.is_contiguous():
        raise ValueError("packed must be contiguous")
    dst = out if out is not None else torch.empty_like(packed)
    _check("cider_int4_from_offset_binary",
           _load().cider_int4_from_offset_binary(_ptr(packed), _ptr(dst), packed.numel(),
                                                 _stream(packed)))
    return dst


def cider_quantize_weight_int8(w: torch.Tensor, group_size: int = 0, clip_percentile=None):
    """w fp32 [N, K] -> (qw int8 [N, K], sw fp32 [N, G]); min-max scales, or
    percentile-clipped ones when ``clip_percentile`` (in (0, 100]) is given."""
    _need(w, torch.float32, "w", 2)
    N, K = w.shape
    G = K // group_size if group_size else 1
    qw = torch.empty((N, K), dtype=torch.int8, device=w.device)
    sw = torch.empty((N, G), dtype=torch.float32, device=w.device)
    if clip_percentile is None:
        _check("cider_quantize_weight_int8",
               _load().cider_quantize_weight_int8(_ptr(w), N, K, group_size, _ptr(qw), _ptr(sw),
                                                  _stream(w)))
    else:
        _check("cider_quantize_weight_int8_clip",
               _load().cider_quantize_weight_int8_clip(_ptr(w), N, K, group_size,
                                                       float(clip_percentile), _ptr(qw), _ptr(sw),
                                                       _stream(w)))
    return qw, sw


def cider_quantize_weight_int4(w: torch.Tensor, group_size: int = 0, clip_percentile=None):
    """w fp32 [N, K] -> (packed uint8 [N, K/2], sw fp32 [N, G]); min-max or
    percentile-clipped scales as for the INT8 quantizer."""
    _need(w, torch.float32, "w", 2)
    N, K = w.shape
    G = K // group_size if group_size else 1
    qp = torch.empty((N, K // 2), dtype=torch.uint8, device=w.device)
    sw = torch.empty((N, G), dtype=torch.float32, device=w.device)
    if clip_percentile is None:
        _check("cider_quantize_weight_int4",
               _load().cider_quantize_weight_int4(_ptr(w), N, K, group_size, _ptr(qp), _ptr(sw),
                                                  _stream(w)))
    else:
        _check("cider_quantize_weight_int4_clip",
               _load().cider_quantize_weight_int4_clip(_ptr(w), N, K, group_size,
                                                       float(clip_percentile), _ptr(qp), _ptr(sw),
                                                       _stream(w)))
    return qp, sw


def _gran(group_size: int) -> int:
    return CIDER_PER_GROUP if group_size else CIDER_PER_CHANNEL


def _linear(fn, x, qw, sw, group_size, int4, out=None, x_dtype=torch.float16):
    _need(x, x_dtype, "x", 2)
    _need(qw, torch.uint8 if int4 else torch.int8, "qw", 2)
    M, K = x.shape
    N = qw.shape[0]
    if qw.shape[1] != (K // 2 if int4 else K):
        raise ValueError("weight width does not match K")
    sw = sw.reshape(N, -1)
    _need(sw, torch.float32, "sw", 2)
    y = out if out is not None else torch.empty((M, N), dtype=torch.float16, device=x.device)
    _check(fn, getattr(_load(), fn)(_ptr(x), M, N, K, _ptr(qw), _ptr(sw), _gran(group_size),
                                    group_size, _ptr(y), _stream(x)))
    return y


def cider_w8a8_linear(x, qw, sw, group_size: int = 0, out=None):
    """y fp16 [M, N] = W8A8 linear of x fp16 [M, K] with qw int8 [N, K] and
    scales sw fp32 [N] (group_size 0) or [N, K/group_size]."""
    return _linear("cider_w8a8_linear", x, qw, sw, group_size, False, out)


def cider_w4a8_linear(x, qw_packed, sw, group_size: int = 0, out=None):
    """W4A8 linear with qw_packed uint8 [N, K/2]."""
    return _linear("cider_w4a8_linear", x, qw_packed, sw, group_size, True, out)


def cider_w8a8_linear_bf16(x, qw, sw, group_size: int = 0, out=None):
    """As cider_w8a8_linear for x bf16 [M, K]; y is fp16."""
    return _linear("cider_w8a8_linear_bf16", x, qw, sw, group_size, False, out, torch.bfloat16)


def cider_w4a8_linear_bf16(x, qw_packed, sw, group_size: int = 0, out=None):
    """As cider_w4a8_linear for x bf16 [M, K]; y is fp16."""
    return _linear("cider_w4a8_linear_bf16", x, qw_packed, sw, group_size, True, out,
                   torch.bfloat16)


def _linear_ex(fn, x, qw, sw, group_size, int4, y_dtype, out):
    if x.dtype not in _DTYPES or y_dtype not in _DTYPES:
        raise TypeError("x and y must be float16 or bfloat16")
    _need(x, x.dtype, "x", 2)
    _need(qw, torch.uint8 if int4 else torch.int8, "qw", 2)
    M, K = x.shape
    N = qw.shape[0]
    if qw.shape[1] != (K // 2 if int4 else K):
        raise ValueError("weight width does not match K")
    sw = sw.reshape(N, -1)
    _need(sw, torch.float32, "sw", 2)
    y = out if out is not None else torch.empty((M, N), dtype=y_dtype, device=x.device)
    _need(y, y_dtype, "out", 2)
    _check(fn, getattr(_load(), fn)(_ptr(x), _DTYPES[x.dtype], M, N, K, _ptr(qw), _ptr(sw),
                                    _gran(group_size), group_size, _ptr(y), _DTYPES[y_dtype],
                                    _stream(x)))
    return y


def cider_w8a8_linear_ex(x, qw, sw, group_size: int = 0, y_dtype=torch.float16, out=None):
    """W8A8 linear with x fp16 or bf16 [M, K] and y of ``y_dtype`` (fp16 or
    bf16, the fp32 result rounded once to it)."""
    return _linear_ex("cider_w8a8_linear_ex", x, qw, sw, group_size, False, y_dtype, out)


def cider_w4a8_linear_ex(x, qw_packed, sw, group_size: int = 0, y_dtype=torch.float16, out=None):
    """W4A8 linear with x fp16 or bf16 [M, K] and y of ``y_dtype``."""
    return _linear_ex("cider_w4a8_linear_ex", x, qw_packed, sw, group_size, True, y_dtype, out)


def _linear_prequant(fn, qa, sa, qw, sw, group_size, int4, out=None):
    _need(qa, torch.int8, "qa", 2)
    _need(sa, torch.float32, "sa", 1)
    _need(qw, torch.uint8 if int4 else torch.int8, "qw", 2)
    M, K = qa.shape
    N = qw.shape[0]
    sw = sw.reshape(N, -1)
    _need(sw, torch.float32, "sw", 2)
    y = out if out is not None else torch.empty((M, N), dtype=torch.float16, device=qa.device)
    _check(fn, getattr(_load(), fn)(_ptr(qa), _ptr(sa), M, N, K, _ptr(qw), _ptr(sw),
                                    _gran(group_size), group_size, _ptr(y), _stream(qa)))
    return y


def cider_w8a8_linear_prequant(qa, sa, qw, sw, group_size: int = 0, out=None):
    return _linear_prequant("cider_w8a8_linear_prequant", qa, sa, qw, sw, group_size, False, out)


def cider_w4a8_linear_prequant(qa, sa, qw_packed, sw, group_size: int = 0, out=None):
    return _linear_prequant("cider_w4a8_linear_prequant", qa, sa, qw_packed, sw, group_size, True,
                            out)


def _accumulators(fn, qa, qw, group_size, int4):
    _need(qa, torch.int8, "qa", 2)
    _need(qw, torch.uint8 if int4 else torch.int8, "qw", 2)
    M, K = qa.shape
    N = qw.shape[0]
    G = K // group_size if group_size else 1
    acc = torch.empty((M, N, G), dtype=torch.int32, device=qa.device)
    _check(fn, getattr(_load(), fn)(_ptr(qa), M, N, K, _ptr(qw), group_size, _ptr(acc),
                                    _stream(qa)))
    return acc


def cider_w8a8_accumulators(qa, qw, group_size: int = 0):
    """Exact int32 accumulators [M, N, G] of the same kernels."""
    return _accumulators("cider_w8a8_accumulators", qa, qw, group_size, False)


def cider_w4a8_accumulators(qa, qw_packed, group_size: int = 0):
    return _accumulators("cider_w4a8_accumulators", qa, qw_packed, group_size, True)


def cider_check_device_error(device=None) -> int:
    """Synchronize the current stream and return (and clear) the status of
    the library's device error word: 0 (CIDER_OK) or 5 (CIDER_ERR_TIMEOUT)."""
    s = torch.cuda.current_stream(device)
    return int(_load().cider_check_device_error(ctypes.c_void_p(s.cuda_stream)))


def cider_trim_scratch_pool(keep_bytes: int = 0, device=None) -> None:
    """Return the library's pooled scratch memory beyond ``keep_bytes`` to the
    device (after the current stream's queued calls have run)."""
    s = torch.cuda.current_stream(device)
    _check("cider_trim_scratch_pool",
           _load().cider_trim_scratch_pool(int(keep_bytes), ctypes.c_void_p(s.cuda_stream)))


def cider_debug_wait_timeout(max_polls: int, device=None) -> int:
    s = torch.cuda.current_stream(device)
    return int(_load().cider_debug_wait_timeout(int(max_polls), ctypes.c_void_p(s.cuda_stream)))


def cider_timing_begin(capacity: int) -> None:
    """Time the integer-GEMM kernel of the next `capacity` linear calls made
    from this thread (CUDA events recorded by the library around each launch)."""
    _check("cider_timing_begin", _load().cider_timing_begin(int(capacity)))


def cider_timing_end():
    """-> (number of timed launches, their summed device time in ms)."""
    n = ctypes.c_int64(0)
    ms = ctypes.c_double(0.0)
    _check("cider_timing_end", _load().cider_timing_end(ctypes.byref(n), ctypes.byref(ms)))
    return int(n.value), float(ms.value)


def cider_debug_pair_schedule(M: int, N: int, K: int, pairs: int):
    """Work split of the per-channel tensor-core GEMM (host arithmetic only).
    -> (info dict, list of (pair, tile, kb0, kb1, kind, row0, row1))."""
    info = (ctypes.c_int32 * 6)()
    count = ctypes.c_int64(0)
    lib = _load()
    _check("cider_debug_pair_schedule",
           lib.cider_debug_pair_schedule(M, N, K, pairs, 0, None, ctypes.byref(count), info))
    rows = (ctypes.c_int32 * (7 * max(count.value, 1)))()
    _check("cider_debug_pair_schedule",
           lib.cider_debug_pair_schedule(M, N, K, pairs, count.value, rows, ctypes.byref(count),
                                         info))
    keys = ("pairs", "whole_tiles", "cut_tiles", "pieces", "blocks_per_tile", "tiles")
    units = [tuple(rows[7 * i:7 * i + 7]) for i in range(count.value)]
    return dict(zip(keys, list(info))), units


def cider_debug_small_m_launch(M: int, N: int, K: int, bits: int, group_size: int,
                               split_allowed: bool, num_sms: int) -> dict:
    """Launch sizes of the small-M path for this linear (host arithmetic only)."""
    info = (ctypes.c_int32 * 10)()
    _check("cider_debug_small_m_launch",
           _load().cider_debug_small_m_launch(M, N, K, 1 if bits == 4 else 0, group_size,
                                              1 if split_allowed else 0, num_sms, info))
    keys = ("mb", "mma", "slices", "tiles_per_slice", "staged_codes", "pitch", "ring_slots",
            "smem", "smem_cap", "codes_per_tile")
    return dict(zip(keys, list(info)))


def cider_debug_small_m_slices(M: int, N: int, K: int, bits: int, group_size: int,
                               num_sms: int) -> int:
    """K slices of the small-M path for this linear (host arithmetic only)."""
    out = ctypes.c_int32(0)
    _check("cider_debug_small_m_slices",
           _load().cider_debug_small_m_slices(M, N, K, 1 if bits == 4 else 0, group_size,
                                              num_sms, ctypes.byref(out)))
    return int(out.value)
