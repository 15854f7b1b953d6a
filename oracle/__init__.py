"""CPU oracle of the W8A8 projection path (test infrastructure only).

Only ``tests/``, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg may import this package.  The product library never loads it, and it
shares no code with the CUDA path.  The arithmetic lives in
``clef_oracle.c`` (plain C, built with ``-ffp-contract=off``); this module
only builds that file and marshals numpy arrays to it.

bf16 tensors are passed as ``uint16`` arrays of bf16 bit patterns, e4m3
tensors as ``uint8`` code arrays.
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "clef_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB = os.path.join(_BUILD, "libclef_oracle.so")
_lock = threading.Lock()
_lib = None

CFLAGS = ["-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared"]


def build(force: bool = False) -> str:
    """Compile the oracle into ``oracle/_build`` (if stale) and return its path."""
    os.makedirs(_BUILD, exist_ok=True)
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".{os.getpid()}.tmp"
        subprocess.check_call(["gcc", *CFLAGS, _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _P(t):
    return C.POINTER(t)


def lib():
    global _lib
    with _lock:
        if _lib is None:
            L = C.CDLL(build())
            i64, u16p, f32p, i8p, u8p = C.c_int64, _P(C.c_uint16), _P(C.c_float), _P(C.c_int8), _P(C.c_uint8)
            L.orc_f32_to_bf16.argtypes = [C.c_float]; L.orc_f32_to_bf16.restype = C.c_uint16
            L.orc_bf16_to_f32.argtypes = [C.c_uint16]; L.orc_bf16_to_f32.restype = C.c_float
            L.orc_f64_to_bf16.argtypes = [C.c_double]; L.orc_f64_to_bf16.restype = C.c_uint16
            L.orc_wht128_f32.argtypes = [f32p]; L.orc_wht128_f32.restype = None
            L.orc_wht128_f64.argtypes = [_P(C.c_double)]; L.orc_wht128_f64.restype = None
            L.orc_rotate_rows_f32.argtypes = [u16p, i64, i64, i64, f32p]
            L.orc_quant_int8_h128.argtypes = [u16p, i64, i64, i64, i8p, f32p]
            L.orc_e4m3_decode.argtypes = [C.c_uint8]; L.orc_e4m3_decode.restype = C.c_double
            L.orc_e4m3_encode.argtypes = [C.c_float]; L.orc_e4m3_encode.restype = C.c_uint8
            L.orc_quant_fp8.argtypes = [u16p, i64, i64, i64, C.c_int, u8p, f32p]
            L.orc_quant_static.argtypes = [u16p, i64, i64, i64, C.c_int, C.c_float, C.c_void_p, f32p]
            L.orc_int8_gemm_acc.argtypes = [i8p, i8p, i64, i64, i64, _P(C.c_int32)]
            L.orc_int8_linear.argtypes = [i8p, f32p, i8p, f32p, u16p, i64, i64, i64, u16p, i64]
            L.orc_swiglu_f32.argtypes = [C.c_float, C.c_float]; L.orc_swiglu_f32.restype = C.c_float
            L.orc_int8_gateup_swiglu.argtypes = [i8p, f32p, i8p, f32p, u16p, i64, i64, i64, u16p, i64]
            L.orc_swiglu_bf16.argtypes = [u16p, i64, i64, i64, u16p, i64]
            L.orc_fp8_linear.argtypes = [u8p, f32p, u8p, f32p, u16p, i64, i64, i64, u16p, i64]
            L.orc_fp8_gateup_swiglu.argtypes = [u8p, f32p, u8p, f32p, u16p, i64, i64, i64, u16p, i64]
            L.orc_lora_t.argtypes = [u16p, i64, u16p, i64, i64, i64, i64, u16p]
            L.orc_lora_y.argtypes = [u16p, u16p, i64, i64, i64, i64, u16p, i64]
            for name in ("orc_rotate_rows_f32", "orc_quant_int8_h128", "orc_quant_fp8",
                         "orc_int8_gemm_acc", "orc_int8_linear", "orc_int8_gateup_swiglu",
                         "orc_swiglu_bf16", "orc_fp8_linear", "orc_fp8_gateup_swiglu", "orc_lora_t", "orc_lora_y"):
                getattr(L, name).restype = C.c_int
            _lib = L
    return _lib


def _ptr(a: np.ndarray, ct):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return a.ctypes.data_as(C.POINTER(ct))


def _check(rc: int, what: str):
    if rc != 0:
        raise RuntimeError(f"oracle {what} failed with code {rc}")


def _c(a, dtype):
    return None if a is None else np.ascontiguousarray(a, dtype=dtype)


# ---------------------------------------------------------------- scalars

def f32_to_bf16(f: float) -> int:
    return int(lib().orc_f32_to_bf16(C.c_float(f)))


def bf16_to_f32(h: int) -> float:
    return float(lib().orc_bf16_to_f32(C.c_uint16(h)))


def f64_to_bf16(d: float) -> int:
    return int(lib().orc_f64_to_bf16(C.c_double(d)))


def e4m3_decode(c: int) -> float:
    return float(lib().orc_e4m3_decode(C.c_uint8(c)))


def e4m3_encode(f: float) -> int:
    return int(lib().orc_e4m3_encode(C.c_float(f)))


def swiglu_f32(g: float, u: float) -> float:
    return float(lib().orc_swiglu_f32(C.c_float(g), C.c_float(u)))


# ---------------------------------------------------------------- rotation

def wht128_f32(v: np.ndarray) -> np.ndarray:
    """Block-128 rotation of one fp32 block (returns a new array)."""
    out = np.array(v, dtype=np.float32, copy=True).reshape(128)
    lib().orc_wht128_f32(_ptr(out, C.c_float))
    return out


def wht128_f64(v: np.ndarray) -> np.ndarray:
    out = np.array(v, dtype=np.float64, copy=True).reshape(128)
    lib().orc_wht128_f64(_ptr(out, C.c_double))
    return out


def rotate_rows(x: np.ndarray) -> np.ndarray:
    """fp32 rotated rows of a bf16 ``[M][K]`` tensor."""
    x = _c(x, np.uint16)
    M, K = x.shape
    out = np.empty((M, K), np.float32)
    _check(lib().orc_rotate_rows_f32(_ptr(x, C.c_uint16), M, K, K, _ptr(out, C.c_float)), "rotate")
    return out


# ---------------------------------------------------------------- quantisers

def quant_int8_h128(x: np.ndarray):
    """(codes int8 [M][K], scales fp32 [M]) of bf16 rows, with block-128 rotation."""
    x = _c(x, np.uint16)
    M, K = x.shape
    q = np.empty((M, K), np.int8)
    s = np.empty(M, np.float32)
    _check(lib().orc_quant_int8_h128(_ptr(x, C.c_uint16), M, K, K, _ptr(q, C.c_int8),
                                     _ptr(s, C.c_float)), "quant_int8_h128")
    return q, s


def quant_fp8(x: np.ndarray, rotate: bool = False):
    """(e4m3 codes uint8 [M][K], scales fp32 [M]) of bf16 rows."""
    x = _c(x, np.uint16)
    M, K = x.shape
    q = np.empty((M, K), np.uint8)
    s = np.empty(M, np.float32)
    _check(lib().orc_quant_fp8(_ptr(x, C.c_uint16), M, K, K, int(rotate), _ptr(q, C.c_uint8),
                               _ptr(s, C.c_float)), "quant_fp8")
    return q, s


def quant_static(x: np.ndarray, s: float, mode: str = "fp8"):
    """(codes [M][K], scales [M] all equal to s) with one static scale s:
    mode "int8_h128" (int8 codes), "fp8" or "fp8_h128" (e4m3 codes as uint8)."""
    x = _c(x, np.uint16)
    M, K = x.shape
    m = {"int8_h128": 0, "fp8": 1, "fp8_h128": 2}[mode]
    q = np.empty((M, K), np.int8 if m == 0 else np.uint8)
    sout = np.empty(M, np.float32)
    _check(lib().orc_quant_static(_ptr(x, C.c_uint16), M, K, K, m, float(np.float32(s)),
                                  q.ctypes.data_as(C.c_void_p), _ptr(sout, C.c_float)), "quant_static")
    return q, sout


# ---------------------------------------------------------------- GEMMs

def int8_gemm_acc(qx: np.ndarray, qw: np.ndarray) -> np.ndarray:
    qx, qw = _c(qx, np.int8), _c(qw, np.int8)
    M, K = qx.shape
    N = qw.shape[0]
    acc = np.empty((M, N), np.int32)
    _check(lib().orc_int8_gemm_acc(_ptr(qx, C.c_int8), _ptr(qw, C.c_int8), M, N, K,
                                   _ptr(acc, C.c_int32)), "int8_gemm_acc")
    return acc


def int8_linear(qx, sx, qw, sw, bias=None) -> np.ndarray:
    qx, qw = _c(qx, np.int8), _c(qw, np.int8)
    sx, sw, bias = _c(sx, np.float32), _c(sw, np.float32), _c(bias, np.uint16)
    M, K = qx.shape
    N = qw.shape[0]
    y = np.empty((M, N), np.uint16)
    _check(lib().orc_int8_linear(_ptr(qx, C.c_int8), _ptr(sx, C.c_float), _ptr(qw, C.c_int8),
                                 _ptr(sw, C.c_float), _ptr(bias, C.c_uint16), M, N, K,
                                 _ptr(y, C.c_uint16), N), "int8_linear")
    return y


def int8_gateup_swiglu(qx, sx, qw_gu, sw_gu, bias_gu=None) -> np.ndarray:
    qx, qw_gu = _c(qx, np.int8), _c(qw_gu, np.int8)
    sx, sw_gu, bias_gu = _c(sx, np.float32), _c(sw_gu, np.float32), _c(bias_gu, np.uint16)
    M, K = qx.shape
    N = qw_gu.shape[0] // 2
    h = np.empty((M, N), np.uint16)
    _check(lib().orc_int8_gateup_swiglu(_ptr(qx, C.c_int8), _ptr(sx, C.c_float),
                                        _ptr(qw_gu, C.c_int8), _ptr(sw_gu, C.c_float),
                                        _ptr(bias_gu, C.c_uint16), M, N, K,
                                        _ptr(h, C.c_uint16), N), "int8_gateup_swiglu")
    return h


def swiglu_bf16(y_gu: np.ndarray) -> np.ndarray:
    y_gu = _c(y_gu, np.uint16)
    M, N2 = y_gu.shape
    N = N2 // 2
    h = np.empty((M, N), np.uint16)
    _check(lib().orc_swiglu_bf16(_ptr(y_gu, C.c_uint16), M, N, N2, _ptr(h, C.c_uint16), N),
           "swiglu_bf16")
    return h


def fp8_linear(qx, sx, qw, sw, bias=None) -> np.ndarray:
    qx, qw = _c(qx, np.uint8), _c(qw, np.uint8)
    sx, sw, bias = _c(sx, np.float32), _c(sw, np.float32), _c(bias, np.uint16)
    M, K = qx.shape
    N = qw.shape[0]
    y = np.empty((M, N), np.uint16)
    _check(lib().orc_fp8_linear(_ptr(qx, C.c_uint8), _ptr(sx, C.c_float), _ptr(qw, C.c_uint8),
                                _ptr(sw, C.c_float), _ptr(bias, C.c_uint16), M, N, K,
                                _ptr(y, C.c_uint16), N), "fp8_linear")
    return y


def fp8_gateup_swiglu(qx, sx, qw_gu, sw_gu, bias_gu=None) -> np.ndarray:
    qx, qw_gu = _c(qx, np.uint8), _c(qw_gu, np.uint8)
    sx, sw_gu, bias_gu = _c(sx, np.float32), _c(sw_gu, np.float32), _c(bias_gu, np.uint16)
    M, K = qx.shape
    N = qw_gu.shape[0] // 2
    h = np.empty((M, N), np.uint16)
    _check(lib().orc_fp8_gateup_swiglu(_ptr(qx, C.c_uint8), _ptr(sx, C.c_float),
                                       _ptr(qw_gu, C.c_uint8), _ptr(sw_gu, C.c_float),
                                       _ptr(bias_gu, C.c_uint16), M, N, K,
                                       _ptr(h, C.c_uint16), N), "fp8_gateup_swiglu")
    return h


# ---------------------------------------------------------------- LoRA

def lora_pad(r: int) -> int:
    """Rank rounded up to a whole 64-group."""
    return (r + 63) // 64 * 64


def lora_t(x, A, r_pad=None) -> np.ndarray:
    x, A = _c(x, np.uint16), _c(A, np.uint16)
    M, K = x.shape
    r = A.shape[0]
    r_pad = lora_pad(r) if r_pad is None else r_pad
    t = np.empty((M, r_pad), np.uint16)
    _check(lib().orc_lora_t(_ptr(x, C.c_uint16), K, _ptr(A, C.c_uint16), M, K, r, r_pad,
                            _ptr(t, C.c_uint16)), "lora_t")
    return t


def lora_y(t, B, y) -> np.ndarray:
    """Returns bf16(y + t B^T) (y is not modified)."""
    t, B = _c(t, np.uint16), _c(B, np.uint16)
    out = np.array(y, dtype=np.uint16, copy=True, order="C")
    M, r_pad = t.shape
    N, r = B.shape
    _check(lib().orc_lora_y(_ptr(t, C.c_uint16), _ptr(B, C.c_uint16), M, N, r, r_pad,
                            _ptr(out, C.c_uint16), N), "lora_y")
    return out


def lora_add(x, A, B, y) -> np.ndarray:
    return lora_y(lora_t(x, A), B, y)
