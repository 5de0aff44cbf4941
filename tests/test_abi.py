"""The C-ABI library builds for sm_103a, loads, exports every entry point that
include/cider.h declares, and rejects bad arguments on the host before any
launch.  No GPU needed: these calls never reach a kernel (bad arguments fail
validation first; calls with well-formed arguments run with
CIDER_FORCE_UNSUPPORTED=1 or on a machine without a GPU, and stop at the
device check)."""
import ctypes
import os
import re
import subprocess

import pytest

from w4a8_quantized_linear_gb300 import _build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "cider.h")

OK, INVALID, MISALIGNED, UNSUPPORTED = 0, 1, 2, 3


@pytest.fixture(scope="module")
def lib():
    path = _build.build()
    import w4a8_quantized_linear_gb300 as pkg
    return pkg.library()


@pytest.fixture
def no_device(monkeypatch):
    monkeypatch.setenv("CIDER_FORCE_UNSUPPORTED", "1")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(cider_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for required in ("cider_quantize_act", "cider_w8a8_linear", "cider_w4a8_linear",
                     "cider_is_available", "cider_w8a8_accumulators"):
        assert required in names


def test_library_exports_every_declared_symbol(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", _build.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = set(re.findall(r"\bT (cider_[a-z0-9_]+)$", out, flags=re.M))
    missing = [n for n in declared_functions() if n not in exported]
    assert not missing, missing
    for n in declared_functions():
        assert getattr(lib, n) is not None


def test_status_strings(lib):
    for s in range(6):
        assert lib.cider_status_string(s)
    assert b"unknown" in lib.cider_status_string(99)
    assert lib.cider_version() >= 100


def test_not_available_without_sm103(lib, no_device):
    assert lib.cider_is_available() == 0


P = 0x10000  # fake, 16-byte aligned "pointer": never dereferenced by these calls


def lin(lib, fn="cider_w8a8_linear", x=P, M=4, N=64, K=256, w=P, sw=P, gran=0, gs=0, y=P):
    return getattr(lib, fn)(x, M, N, K, w, sw, gran, gs, y, None)


def test_empty_problem_is_a_noop(lib):
    assert lin(lib, M=0, x=None, w=None, sw=None, y=None) == OK
    assert lin(lib, N=0, x=None, w=None, sw=None, y=None) == OK
    assert lib.cider_quantize_act(None, 0, 256, None, None, None) == OK
    assert lib.cider_w8a8_accumulators(None, 0, 8, 64, None, 0, None, None) == OK


@pytest.mark.parametrize("kw", [
    dict(x=None), dict(w=None), dict(sw=None), dict(y=None),
    dict(M=-1), dict(N=-8), dict(K=0), dict(K=16), dict(K=48), dict(K=200000),
    dict(N=12),                         # N % 8
    dict(gran=0, gs=64),                # per channel with a group size
    dict(gran=1, gs=0), dict(gran=1, gs=32), dict(gran=1, gs=256),
    dict(gran=1, gs=128, K=192),        # K % gs
    dict(gran=7),
])
@pytest.mark.parametrize("fn", ["cider_w8a8_linear", "cider_w4a8_linear"])
def test_invalid_arguments(lib, no_device, fn, kw):
    assert lin(lib, fn=fn, **kw) == INVALID


@pytest.mark.parametrize("kw", [dict(x=P + 8), dict(w=P + 4), dict(y=P + 2), dict(sw=P + 2)])
def test_misaligned(lib, no_device, kw):
    assert lin(lib, **kw) == MISALIGNED


def test_well_formed_call_stops_at_device_check(lib, no_device):
    assert lin(lib) == UNSUPPORTED
    assert lin(lib, fn="cider_w4a8_linear", gran=1, gs=128) == UNSUPPORTED
    assert lib.cider_quantize_act(P, 4, 256, P, P, None) == UNSUPPORTED
    assert lib.cider_quantize_weight_int8(P, 8, 256, 64, P, P, None) == UNSUPPORTED
    assert lib.cider_quantize_weight_int4(P, 8, 256, 0, P, P, None) == UNSUPPORTED
    assert lib.cider_w8a8_linear_prequant(P, P, 4, 64, 256, P, P, 1, 64, P, None) == UNSUPPORTED
    assert lib.cider_w8a8_accumulators(P, 4, 64, 256, P, 128, P, None) == UNSUPPORTED
    assert lib.cider_check_device_error(None) == UNSUPPORTED
    assert lib.cider_debug_wait_timeout(10, None) == UNSUPPORTED


def test_quantize_and_prequant_argument_checks(lib, no_device):
    assert lib.cider_quantize_act(P, 4, 100, P, P, None) == INVALID
    assert lib.cider_quantize_act(P + 8, 4, 256, P, P, None) == MISALIGNED
    assert lib.cider_quantize_act(P, 4, 256, P, P + 1, None) == MISALIGNED
    assert lib.cider_quantize_weight_int8(P, 8, 256, 96, P, P, None) == INVALID
    assert lib.cider_quantize_weight_int4(P, 8, 96, 64, P, P, None) == INVALID
    assert lib.cider_w8a8_linear_prequant(None, P, 4, 64, 256, P, P, 0, 0, P, None) == INVALID
    assert lib.cider_w8a8_linear_prequant(P, None, 4, 64, 256, P, P, 0, 0, P, None) == INVALID
    assert lib.cider_w8a8_accumulators(P, 4, 64, 256, P, 96, P, None) == INVALID
    assert lib.cider_w4a8_accumulators(P, 4, 64, 256, P, 0, None, None) == INVALID
    assert lib.cider_debug_wait_timeout(0, None) == INVALID


def test_binding_fails_loudly_without_library(monkeypatch):
    import w4a8_quantized_linear_gb300 as pkg
    monkeypatch.setattr(pkg, "_lib", None)
    monkeypatch.setattr(pkg, "LIB_PATH", "/nonexistent/libcider.so")
    with pytest.raises(RuntimeError, match="no fallback"):
        pkg.library()


def test_timing_argument_checks(lib):
    assert lib.cider_timing_begin(0) == INVALID
    assert lib.cider_timing_end(None, None) == INVALID


@pytest.mark.parametrize("fn", ["cider_w8a8_linear_bf16", "cider_w4a8_linear_bf16"])
def test_bf16_linears_check_like_the_fp16_ones(lib, no_device, fn):
    assert lin(lib, fn=fn) == UNSUPPORTED
    assert lin(lib, fn=fn, x=None) == INVALID
    assert lin(lib, fn=fn, N=12) == INVALID
    assert lin(lib, fn=fn, gran=1, gs=32) == INVALID
    assert lin(lib, fn=fn, x=P + 8) == MISALIGNED
    assert lin(lib, fn=fn, M=0, x=None, w=None, sw=None, y=None) == OK


def test_bf16_quantize_and_int4_import_argument_checks(lib, no_device):
    assert lib.cider_quantize_act_bf16(P, 4, 256, P, P, None) == UNSUPPORTED
    assert lib.cider_quantize_act_bf16(P, 4, 100, P, P, None) == INVALID
    assert lib.cider_quantize_act_bf16(P + 8, 4, 256, P, P, None) == MISALIGNED
    assert lib.cider_quantize_act_bf16(None, 0, 256, None, None, None) == OK
    assert lib.cider_int4_from_offset_binary(P, P, 1000, None) == UNSUPPORTED
    assert lib.cider_int4_from_offset_binary(P, P, 0, None) == OK
    assert lib.cider_int4_from_offset_binary(P, P, -1, None) == INVALID
    assert lib.cider_int4_from_offset_binary(None, P, 16, None) == INVALID
    assert lib.cider_int4_from_offset_binary(P + 4, P, 16, None) == MISALIGNED


def test_debug_split_queries_need_no_device(lib):
    n = ctypes.c_int64(0)
    info = (ctypes.c_int32 * 6)()
    assert lib.cider_debug_pair_schedule(4096, 10240, 2560, 76, 0, None, ctypes.byref(n), info) == OK
    assert n.value > 0 and info[0] == 76
    ks = ctypes.c_int32(0)
    assert lib.cider_debug_small_m_slices(16, 2560, 10240, 0, 0, 152, ctypes.byref(ks)) == OK
    assert ks.value > 1
    assert lib.cider_debug_small_m_slices(0, 2560, 10240, 0, 0, 152, ctypes.byref(ks)) == INVALID


def test_dtype_linears_and_clipped_quantizers_check_arguments(lib, no_device):
    """The dtype-aware linears and the percentile-clipped weight quantizers:
    bad dtypes and percentiles are rejected, well-formed calls stop at the
    device check (no GPU involved)."""
    for fn in ("cider_w8a8_linear_ex", "cider_w4a8_linear_ex"):
        f = getattr(lib, fn)
        assert f(P, 0, 4, 64, 256, P, P, 0, 0, P, 1, None) == UNSUPPORTED
        assert f(P, 1, 4, 64, 256, P, P, 1, 128, P, 0, None) == UNSUPPORTED
        assert f(P, 2, 4, 64, 256, P, P, 0, 0, P, 0, None) == INVALID      # unknown x dtype
        assert f(P, 0, 4, 64, 256, P, P, 0, 0, P, -1, None) == INVALID     # unknown y dtype
        assert f(None, 0, 4, 64, 256, P, P, 0, 0, P, 1, None) == INVALID
        assert f(P, 0, 4, 64, 100, P, P, 0, 0, P, 1, None) == INVALID      # K % 32
        assert f(P + 8, 0, 4, 64, 256, P, P, 0, 0, P, 1, None) == MISALIGNED
        assert f(P, 0, 0, 64, 256, P, P, 0, 0, P, 1, None) == 0              # empty problem
    for fn in ("cider_quantize_weight_int8_clip", "cider_quantize_weight_int4_clip"):
        f = getattr(lib, fn)
        assert f(P, 8, 256, 64, 99.9, P, P, None) == UNSUPPORTED
        assert f(P, 8, 256, 0, 100.0, P, P, None) == UNSUPPORTED
        for bad in (0.0, -1.0, 100.5, float("nan")):
            assert f(P, 8, 256, 64, bad, P, P, None) == INVALID
        assert f(P, 8, 256, 96, 99.9, P, P, None) == INVALID                 # group size
        assert f(P + 1, 8, 256, 0, 99.9, P, P, None) == MISALIGNED


def test_trim_scratch_pool_argument_checks(lib, no_device):
    assert lib.cider_trim_scratch_pool(-1, None) == INVALID
    assert lib.cider_trim_scratch_pool(0, None) == UNSUPPORTED
