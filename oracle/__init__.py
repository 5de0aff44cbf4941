"""CPU oracle for the W8A8 / W4A8 online-activation-quantized linear layer.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package.  The product library
(``w4a8_quantized_linear_gb300``) never imports it and shares no code with it.

The arithmetic lives in ``cider_oracle.c`` (plain single-threaded C, built with
``-O2 -ffp-contract=off``); this module only builds it with gcc and marshals
numpy arrays through ctypes.  Each function names the passage of the Cider
README (page "cider") it follows; the C file states the readings taken where
the page is silent.

Parity status: every function here is pinned by ``tests/test_oracle_pins.py``
(hand-worked cases, exhaustive enumeration, brute force and closed forms).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from concurrent.futures import ThreadPoolExecutor

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "cider_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libcider_oracle.so")
_CFLAGS = ["-O2", "-ffp-contract=off", "-fno-fast-math", "-std=c11", "-fPIC", "-shared"]

_lib = None
_lock = threading.Lock()


def build(force: bool = False) -> str:
    """Compile the oracle with gcc into ``oracle/_build`` and return the path."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    hdr = os.path.join(_HERE, "cider_oracle.h")
    stale = (not os.path.exists(_LIB_PATH)) or any(
        os.path.getmtime(p) > os.path.getmtime(_LIB_PATH) for p in (_SRC, hdr))
    if force or stale:
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", *_CFLAGS, "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _configure(lib):
    """Declare the C signatures on a loaded oracle library."""
    i64, p = ctypes.c_int64, ctypes.c_void_p
    lib.oracle_f16_to_f32.argtypes = [ctypes.c_uint16]
    lib.oracle_f16_to_f32.restype = ctypes.c_float
    lib.oracle_f32_to_f16.argtypes = [ctypes.c_float]
    lib.oracle_f32_to_f16.restype = ctypes.c_uint16
    lib.oracle_f32_to_bf16.argtypes = [ctypes.c_float]
    lib.oracle_f32_to_bf16.restype = ctypes.c_uint16
    lib.oracle_quantize_weight_int8_clip.argtypes = [p, i64, i64, i64, ctypes.c_double, p, p, p]
    lib.oracle_quantize_weight_int4_clip.argtypes = [p, i64, i64, i64, ctypes.c_double, p, p, p]
    lib.oracle_dequant_pc_bf16.argtypes = [p, p, p, i64, i64, p]
    lib.oracle_dequant_pg_bf16.argtypes = [p, p, p, i64, i64, i64, p]
    lib.oracle_linear_rows_ex.argtypes = [p, ctypes.c_int, i64, i64, p, p, i64, i64, i64, p, p,
                                          ctypes.c_int, p]
    lib.oracle_linear_rows_ex.restype = ctypes.c_int
    lib.oracle_quantize_act.argtypes = [p, i64, i64, p, p]
    lib.oracle_quantize_act_bf16.argtypes = [p, i64, i64, p, p]
    lib.oracle_int4_from_offset_binary.argtypes = [p, i64, p]
    lib.oracle_linear_rows_bf16.argtypes = [p, i64, i64, p, p, i64, i64, i64, p, p, p]
    lib.oracle_linear_rows_bf16.restype = ctypes.c_int
    lib.oracle_quantize_weight_int8.argtypes = [p, i64, i64, i64, p, p]
    lib.oracle_quantize_weight_int4.argtypes = [p, i64, i64, i64, p, p]
    lib.oracle_pack_int4.argtypes = [p, i64, i64, p]
    lib.oracle_unpack_int4.argtypes = [p, i64, i64, p]
    lib.oracle_gemm_acc.argtypes = [p, p, i64, i64, i64, i64, p]
    lib.oracle_gemm_acc.restype = ctypes.c_int
    lib.oracle_dequant_pc.argtypes = [p, p, p, i64, i64, p]
    lib.oracle_dequant_pg.argtypes = [p, p, p, i64, i64, i64, p]
    lib.oracle_linear_rows.argtypes = [p, i64, i64, p, p, i64, i64, i64, p, p, p]
    lib.oracle_linear_rows.restype = ctypes.c_int
    return lib


def _load():
    global _lib
    with _lock:
        if _lib is None:
            _lib = _configure(ctypes.CDLL(build()))
    return _lib


def _c(a: np.ndarray, dtype) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=dtype)


def _ptr(a: np.ndarray) -> int:
    return a.ctypes.data


def f16_bits(x: np.ndarray) -> np.ndarray:
    """fp16 array -> its uint16 bit patterns (a view; no arithmetic)."""
    return _c(x, np.float16).view(np.uint16)


# ---------------------------------------------------------------- a1
def quantize_act(x_f16: np.ndarray, threads: int = 1):
    """Per-token symmetric INT8 quantization (Cider README, "Metal kernel
    pipeline": quantize_per_token; "Quantization": activations per token).
    x fp16 [M,K] -> (qa int8 [M,K], sa fp32 [M]).  Rows are independent, so
    ``threads > 1`` runs disjoint row ranges of the same single-threaded C
    code concurrently (ctypes releases the GIL)."""
    x = f16_bits(x_f16)
    M, K = x.shape
    qa = np.empty((M, K), np.int8)
    sa = np.empty((M,), np.float32)
    lib = _load()

    def run(r0, r1):
        r0, r1 = int(r0), int(r1)
        lib.oracle_quantize_act(_ptr(x) + r0 * K * 2, r1 - r0, K, _ptr(qa) + r0 * K,
                                _ptr(sa) + r0 * 4)

    if threads <= 1 or M < 2:
        run(0, M)
    else:
        bounds = np.linspace(0, M, min(threads, M) + 1).astype(int)
        with ThreadPoolExecutor(len(bounds) - 1) as ex:
            list(ex.map(lambda i: run(bounds[i], bounds[i + 1]), range(len(bounds) - 1)))
    return qa, sa


def quantize_act_bf16(x_bf16_bits: np.ndarray):
    """The same for bf16 activations, given as their uint16 bit patterns
    [M,K] (numpy has no bf16 type): each widens exactly to fp32 (the README's
    roadmap, "auto dtype float16/bfloat16")."""
    x = _c(x_bf16_bits, np.uint16)
    M, K = x.shape
    qa = np.empty((M, K), np.int8)
    sa = np.empty((M,), np.float32)
    _load().oracle_quantize_act_bf16(_ptr(x), M, K, _ptr(qa), _ptr(sa))
    return qa, sa


def int4_from_offset_binary(src: np.ndarray) -> np.ndarray:
    """uint8 bytes of offset-binary INT4 (nibble u holds u - 8; README
    "Quantization": "Symmetric INT4 (zp=8)") -> the two's complement packing
    of the same values, nibble order unchanged."""
    src = _c(src, np.uint8)
    dst = np.empty_like(src)
    _load().oracle_int4_from_offset_binary(_ptr(src), src.size, _ptr(dst))
    return dst


# ---------------------------------------------------------------- a2 / a4
def quantize_weight_int8(W: np.ndarray, group_size: int = 0, clip_percentile=None):
    """Symmetric INT8 weights, per channel (group_size=0) or per group
    (Cider README, "Quantization" and "W8A8 quantization granularity"), with
    min-max scales or, given ``clip_percentile`` in (0, 100], percentile-clipped
    ones ("Notes": clip_percentile=99.9; definition in cider_oracle.c).
    W fp32 [N,K] -> (qw int8 [N,K], sw fp32 [N,G])."""
    W = _c(W, np.float32)
    N, K = W.shape
    G = K // group_size if group_size else 1
    qw = np.empty((N, K), np.int8)
    sw = np.empty((N, G), np.float32)
    if clip_percentile is None:
        _load().oracle_quantize_weight_int8(_ptr(W), N, K, group_size, _ptr(qw), _ptr(sw))
    else:
        tmp = np.empty((K,), np.float32)
        _load().oracle_quantize_weight_int8_clip(_ptr(W), N, K, group_size, float(clip_percentile),
                                                 _ptr(qw), _ptr(sw), _ptr(tmp))
    return qw, sw


def quantize_weight_int4(W: np.ndarray, group_size: int = 0, clip_percentile=None):
    """Symmetric INT4 weights in [-8,7] with s = max|W|/7 (or the clipped
    percentile / 7).  W fp32 [N,K] -> (q4 int8 [N,K] values, sw fp32 [N,G])."""
    W = _c(W, np.float32)
    N, K = W.shape
    G = K // group_size if group_size else 1
    q4 = np.empty((N, K), np.int8)
    sw = np.empty((N, G), np.float32)
    if clip_percentile is None:
        _load().oracle_quantize_weight_int4(_ptr(W), N, K, group_size, _ptr(q4), _ptr(sw))
    else:
        tmp = np.empty((K,), np.float32)
        _load().oracle_quantize_weight_int4_clip(_ptr(W), N, K, group_size, float(clip_percentile),
                                                 _ptr(q4), _ptr(sw), _ptr(tmp))
    return q4, sw


def pack_int4(q4: np.ndarray) -> np.ndarray:
    """[N,K] values in [-8,7] -> uint8 [N,K/2], element 2j in the low nibble."""
    q4 = _c(q4, np.int8)
    N, K = q4.shape
    out = np.empty((N, K // 2), np.uint8)
    _load().oracle_pack_int4(_ptr(q4), N, K, _ptr(out))
    return out


def unpack_int4(packed: np.ndarray) -> np.ndarray:
    """uint8 [N,K/2] -> int8 [N,K] two's complement nibble values."""
    packed = _c(packed, np.uint8)
    N, Kh = packed.shape
    out = np.empty((N, 2 * Kh), np.int8)
    _load().oracle_unpack_int4(_ptr(packed), N, 2 * Kh, _ptr(out))
    return out


# ---------------------------------------------------------------- a3
def gemm_acc(qa: np.ndarray, qw: np.ndarray, group_size: int = 0) -> np.ndarray:
    """INT32 accumulators [M,N,G] of qa [M,K] x qw[N,K]^T (Cider README,
    "Quantization": INT32 accumulation).  Raises if a sum overflows int32."""
    qa = _c(qa, np.int8)
    qw = _c(qw, np.int8)
    M, K = qa.shape
    N = qw.shape[0]
    G = K // group_size if group_size else 1
    acc = np.empty((M, N, G), np.int32)
    if _load().oracle_gemm_acc(_ptr(qa), _ptr(qw), M, N, K, group_size, _ptr(acc)) != 0:
        raise OverflowError("integer accumulator does not fit in int32")
    return acc


# ---------------------------------------------------------------- a5
def dequant_pc(acc: np.ndarray, sa: np.ndarray, sw: np.ndarray, bf16: bool = False) -> np.ndarray:
    """y = round((float(acc) * s_a) * s_w) (Cider README, "Quantization":
    output dequant) to fp16, or with ``bf16`` to bf16 (returned as uint16 bit
    patterns).  acc [M,N] or [M,N,1] -> [M,N]."""
    acc = _c(acc, np.int32)
    M, N = acc.shape[0], acc.shape[1]
    sa = _c(sa, np.float32)
    sw = _c(sw, np.float32)
    y = np.empty((M, N), np.uint16)
    fn = _load().oracle_dequant_pc_bf16 if bf16 else _load().oracle_dequant_pc
    fn(_ptr(acc), _ptr(sa), _ptr(sw), M, N, _ptr(y))
    return y if bf16 else y.view(np.float16)


def dequant_pg(acc: np.ndarray, sa: np.ndarray, sw: np.ndarray, bf16: bool = False) -> np.ndarray:
    """y = round(sum_g in increasing g of (s_a * s_w[n,g]) * float(acc_g)) to
    fp16 (or bf16 bit patterns).  acc [M,N,G], sw [N,G] -> [M,N]."""
    acc = _c(acc, np.int32)
    M, N, G = acc.shape
    sa = _c(sa, np.float32)
    sw = _c(sw, np.float32)
    y = np.empty((M, N), np.uint16)
    fn = _load().oracle_dequant_pg_bf16 if bf16 else _load().oracle_dequant_pg
    fn(_ptr(acc), _ptr(sa), _ptr(sw), M, N, G, _ptr(y))
    return y if bf16 else y.view(np.float16)


# ---------------------------------------------------------------- whole layer
def linear(x_f16: np.ndarray, qw_values: np.ndarray, sw: np.ndarray,
           group_size: int = 0, rows=None, threads: int = 1, bf16: bool = False,
           out_bf16: bool = False) -> np.ndarray:
    """The whole layer, y [len(rows), N], for the given activation rows
    (default: all).  ``qw_values`` holds the integer weight values (INT8, or
    INT4 values from :func:`unpack_int4`).  With ``bf16`` the activations are
    bf16 bit patterns (uint16 [M,K]); with ``out_bf16`` y is rounded to bf16
    and returned as uint16 bit patterns (else fp16).  Rows are independent, so
    ``threads > 1`` runs disjoint row ranges of the same single-threaded C
    code concurrently (ctypes releases the GIL)."""
    x = _c(x_f16, np.uint16) if bf16 else f16_bits(x_f16)
    M, K = x.shape
    qw = _c(qw_values, np.int8)
    N = qw.shape[0]
    sw = _c(sw, np.float32)
    G = K // group_size if group_size else 1
    rows = np.arange(M) if rows is None else np.asarray(rows, dtype=np.int64)
    xs = np.ascontiguousarray(x[rows])
    R = xs.shape[0]
    y = np.empty((R, N), np.uint16)
    lib = _load()

    def run(r0, r1):
        qa_s = np.empty((K,), np.int8)
        acc_s = np.empty((max(N * G, 1),), np.int32)
        r0, r1 = int(r0), int(r1)
        st = lib.oracle_linear_rows_ex(_ptr(xs), 1 if bf16 else 0, K, N, _ptr(qw), _ptr(sw),
                                       group_size, r0, r1, _ptr(qa_s), _ptr(acc_s),
                                       1 if out_bf16 else 0, _ptr(y) + r0 * N * 2)
        if st != 0:
            raise OverflowError("integer accumulator does not fit in int32")

    if threads <= 1 or R < 2:
        run(0, R)
    else:
        bounds = np.linspace(0, R, min(threads, R) + 1).astype(int)
        with ThreadPoolExecutor(len(bounds) - 1) as ex:
            list(ex.map(lambda i: run(bounds[i], bounds[i + 1]), range(len(bounds) - 1)))
    return y if out_bf16 else y.view(np.float16)


def f32_to_bf16(v: float) -> int:
    """bf16 bit pattern of fp32 v, round to nearest even (the oracle's output
    rounding for bf16 y)."""
    return int(_load().oracle_f32_to_bf16(v))


def f16_to_f32(bits: int) -> float:
    return float(_load().oracle_f16_to_f32(bits))


def f32_to_f16(v: float) -> int:
    return int(_load().oracle_f32_to_f16(v))
