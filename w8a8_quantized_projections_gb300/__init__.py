"""Python binding of the GB300 W8A8 quantized projection library (libclef.so).

Argument marshalling only: every function checks tensor placement, dtype and
layout, allocates outputs with torch when the caller passes none, and calls
the C ABI of ``include/clef.h`` on the current CUDA stream.  All arithmetic
runs in the library's CUDA kernels; there is no fallback path, and a missing
library or GPU raises.

bf16 tensors are ``torch.bfloat16``; INT8 codes ``torch.int8``; e4m3 codes
``torch.uint8`` (bit patterns; ``torch.float8_e4m3fn`` inputs are accepted).
"""
from __future__ import annotations

import ctypes as C
import os
import threading

import torch

from . import build as _build

__all__ = [
    "ClefError", "library", "library_path", "quant_act", "quant_act_static", "w8a8_linear", "w8a8_gateup_swiglu",
    "fp8_linear", "fp8_gateup_swiglu", "lora_add", "lora_add_noalloc", "lora_shrink", "lora_expand_add",
    "lora_gateup_swiglu", "swiglu_bf16",
    "w8a8_gemm_s32", "w8a8_linear_lora", "w8a8_gateup_swiglu_lora",
    "poll_status", "set_wait_limit_ns", "set_quant_staging", "set_pdl", "ACT_MODES", "gemm_workspace_bytes",
    "bind_workspace", "mma_peak",
]

ACT_MODES = {"int8_h128": 0, "fp8": 1, "fp8_h128": 2}
_STATUS = {0: "CLEF_OK", 1: "CLEF_ERR_INVALID_ARG", 2: "CLEF_ERR_UNSUPPORTED", 3: "CLEF_ERR_CUDA",
           4: "CLEF_ERR_TIMEOUT"}

_lock = threading.Lock()
_lib = None


class ClefError(RuntimeError):
    def __init__(self, call: str, status: int, detail: str = ""):
        self.status = status
        super().__init__(f"{call} returned {_STATUS.get(status, status)}" + (f": {detail}" if detail else ""))


def library_path() -> str:
    return _build.LIB


def library():
    """The loaded libclef.so (built on first use if absent or stale)."""
    global _lib
    with _lock:
        if _lib is None:
            path = _build.build()
            if not os.path.exists(path):
                raise RuntimeError(f"CUDA library missing at {path}")
            L = C.CDLL(path)
            vp, i64, i32 = C.c_void_p, C.c_int64, C.c_int
            sigs = {
                "clef_quant_act": [vp, i64, i64, i64, i32, vp, vp, vp],
                "clef_quant_act_static": [vp, i64, i64, i64, i32, C.c_float, vp, vp, vp],
                "clef_w8a8_linear": [vp, vp, vp, vp, vp, i64, i64, i64, vp, i64, vp],
                "clef_w8a8_gateup_swiglu": [vp, vp, vp, vp, vp, i64, i64, i64, vp, i64, vp],
                "clef_fp8_linear": [vp, vp, vp, vp, vp, i64, i64, i64, vp, i64, vp],
                "clef_fp8_gateup_swiglu": [vp, vp, vp, vp, vp, i64, i64, i64, vp, i64, vp],
                "clef_lora_add": [vp, i64, vp, vp, i64, i64, i64, i64, vp, vp, i64, vp],
                "clef_lora_add_noalloc": [vp, i64, vp, vp, i64, i64, i64, i64, vp, i64, vp],
                "clef_lora_shrink": [vp, i64, vp, i64, i64, i64, vp, i64, vp],
                "clef_gemm_workspace_bytes": [vp],
                "clef_bind_workspace": [vp, vp, i64],
                "clef_lora_expand_add": [vp, i64, vp, i64, i64, i64, vp, i64, vp],
                "clef_swiglu_bf16": [vp, i64, i64, i64, vp, i64, vp],
                "clef_lora_gateup_swiglu": [vp, i64, vp, vp, vp, vp, i64, i64, i64, i64, vp, vp, i64,
                                            vp, i64, vp],
                "clef_w8a8_gemm_s32": [vp, vp, i64, i64, i64, vp, i64, vp],
                "clef_w8a8_linear_lora": [vp, vp, vp, vp, vp, i64, i64, i64, vp, i64, vp, i64, i32, vp, vp,
                                          vp, i64, vp],
                "clef_w8a8_gateup_swiglu_lora": [vp, vp, vp, vp, vp, i64, i64, i64, vp, i64, vp, vp, i64, vp,
                                                 i64, vp],
                "clef_mma_peak": [i32, i64, vp],
                "clef_set_sm_budget": [i32],
                "clef_copy_sm": [vp, vp, i64, i32, vp],
                "clef_poll_status": [],
                "clef_abi_version": [],
            }
            for name, args in sigs.items():
                fn = getattr(L, name)
                fn.argtypes = args
                fn.restype = C.c_int
            L.clef_set_wait_limit_ns.argtypes = [C.c_uint64]
            L.clef_set_wait_limit_ns.restype = None
            L.clef_status_string.argtypes = [C.c_int]
            L.clef_status_string.restype = C.c_char_p
            L.clef_last_error.argtypes = []
            L.clef_last_error.restype = C.c_char_p
            _lib = L
    return _lib


def _call(name: str, *args) -> None:
    L = library()
    rc = getattr(L, name)(*args)
    if rc != 0:
        raise ClefError(name, rc, L.clef_last_error().decode(errors="replace"))


def _stream(t: torch.Tensor, stream=None):
    s = stream if stream is not None else torch.cuda.current_stream(t.device)
    return C.c_void_p(s.cuda_stream)


def _cuda(t: torch.Tensor, name: str, dtypes) -> torch.Tensor:
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype not in dtypes:
        raise ValueError(f"{name} has dtype {t.dtype}, expected one of {dtypes}")
    return t


def _rows(t: torch.Tensor, name: str) -> int:
    """Row pitch of a 2-D tensor whose rows are contiguous."""
    if t.dim() != 2 or t.stride(1) != 1:
        raise ValueError(f"{name} must be 2-D with contiguous rows")
    return t.stride(0) if t.size(0) > 1 else t.size(1)


def _dense(t: torch.Tensor, name: str) -> torch.Tensor:
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t


def _ptr(t):
    return C.c_void_p(t.data_ptr()) if t is not None else C.c_void_p(None)


_FP8 = (torch.uint8, torch.float8_e4m3fn)


def quant_act(x: torch.Tensor, mode: str = "int8_h128", q=None, scale=None, stream=None):
    """Per-token quantizer: returns (codes [M][K], scales fp32 [M])."""
    _cuda(x, "x", (torch.bfloat16,))
    ldx = _rows(x, "x")
    M, K = x.shape
    m = ACT_MODES[mode]
    if q is None:
        q = torch.empty((M, K), dtype=torch.int8 if m == 0 else torch.uint8, device=x.device)
    if scale is None:
        scale = torch.empty((M,), dtype=torch.float32, device=x.device)
    _dense(q, "q")
    _call("clef_quant_act", _ptr(x), M, K, ldx, m, _ptr(q), _ptr(scale), _stream(x, stream))
    return q, scale


def quant_act_static(x: torch.Tensor, s: float, mode: str = "fp8", q=None, scale=None, stream=None):
    """Quantizer with one static scale s for every row: returns (codes, scales = s)."""
    _cuda(x, "x", (torch.bfloat16,))
    ldx = _rows(x, "x")
    M, K = x.shape
    m = ACT_MODES[mode]
    if q is None:
        q = torch.empty((M, K), dtype=torch.int8 if m == 0 else torch.uint8, device=x.device)
    if scale is None:
        scale = torch.empty((M,), dtype=torch.float32, device=x.device)
    _dense(q, "q")
    _call("clef_quant_act_static", _ptr(x), M, K, ldx, m, float(s), _ptr(q), _ptr(scale), _stream(x, stream))
    return q, scale


def _w8a8(name, codes, qx, sx, qw, sw, bias, out, n_out, stream):
    _w8a8_checks(codes, qx, sx, qw, sw, bias)
    M, K = qx.shape
    if out is None:
        out = torch.empty((M, n_out), dtype=torch.bfloat16, device=qx.device)
    _cuda(out, "out", (torch.bfloat16,))
    _out_shape(out, M, n_out)
    ldo = _rows(out, "out")
    _call(name, _ptr(qx), _ptr(sx), _ptr(qw), _ptr(sw), _ptr(bias), M, n_out, K, _ptr(out), ldo,
          _stream(qx, stream))
    return out


def _out_shape(out, M, n_out):
    # the kernels write M rows of n_out columns at the output's pitch
    if tuple(out.shape) != (M, n_out):
        raise ValueError(f"output has shape {tuple(out.shape)}, expected ({M}, {n_out})")


def _w8a8_checks(codes, qx, sx, qw, sw, bias):
    """The library takes bare pointers and cannot check buffer lengths, so
    they are checked here: a short scale or bias vector would be read past
    its end by the epilogue."""
    _cuda(qx, "qx", codes)
    _cuda(qw, "qw", codes)
    _dense(qx, "qx"); _dense(qw, "qw")
    if qx.dim() != 2 or qw.dim() != 2:
        raise ValueError("qx and qw must be 2-D")
    _cuda(sx, "sx", (torch.float32,)); _cuda(sw, "sw", (torch.float32,))
    _dense(sx, "sx"); _dense(sw, "sw")
    M, K = qx.shape
    rows = qw.shape[0]
    if qw.shape[1] != K:
        raise ValueError("qx and qw disagree on K")
    if sx.numel() != M:
        raise ValueError(f"sx has {sx.numel()} values for {M} rows of qx")
    if sw.numel() != rows:
        raise ValueError(f"sw has {sw.numel()} values for {rows} weight rows")
    if bias is not None:
        _cuda(bias, "bias", (torch.bfloat16,))
        _dense(bias, "bias")
        if bias.numel() != rows:
            raise ValueError(f"bias has {bias.numel()} values for {rows} weight rows")


def w8a8_linear(qx, sx, qw, sw, bias=None, y=None, stream=None):
    """y = bf16(((acc * sx) * sw) + bias) with acc the exact INT8 GEMM of qx and qw^T."""
    return _w8a8("clef_w8a8_linear", (torch.int8,), qx, sx, qw, sw, bias, y, qw.shape[0], stream)


def _gateup_half(qw_gu) -> int:
    if qw_gu.dim() != 2 or qw_gu.shape[0] % 2 != 0:
        raise ValueError("packed gate/up weights need an even row count (gate rows, then up rows)")
    return qw_gu.shape[0] // 2


def w8a8_gateup_swiglu(qx, sx, qw_gu, sw_gu, bias_gu=None, h=None, stream=None):
    """h = bf16(silu(g) * u) for packed gate/up INT8 weights [2N][K]."""
    _gateup_half(qw_gu)
    return _w8a8("clef_w8a8_gateup_swiglu", (torch.int8,), qx, sx, qw_gu, sw_gu, bias_gu, h,
                 qw_gu.shape[0] // 2, stream)


def fp8_linear(qx, sx, qw, sw, bias=None, y=None, stream=None):
    return _w8a8("clef_fp8_linear", _FP8, qx, sx, qw, sw, bias, y, qw.shape[0], stream)


def fp8_gateup_swiglu(qx, sx, qw_gu, sw_gu, bias_gu=None, h=None, stream=None):
    _gateup_half(qw_gu)
    return _w8a8("clef_fp8_gateup_swiglu", _FP8, qx, sx, qw_gu, sw_gu, bias_gu, h,
                 qw_gu.shape[0] // 2, stream)


def _lora_t(t, B, r_cols, M):
    _cuda(t, "t", (torch.bfloat16,))
    _cuda(B, "B", (torch.bfloat16,))
    _dense(B, "B")
    if t.dim() != 2 or t.shape[0] != M or t.shape[1] < r_cols:
        raise ValueError(f"t must have {M} rows and at least {r_cols} columns")
    return _rows(t, "t")


def w8a8_linear_lora(qx, sx, qw, sw, bias, t, B, y=None, segments=None, stream=None):
    """INT8 linear with the LoRA expand fused: y = bf16(bf16(linear) + t B^T),
    the bytes of w8a8_linear followed by lora_expand_add.  t: bf16 [M][>= r_pad]
    from lora_shrink; B: bf16 [N][r] (adapters stacked in output order for a
    packed projection).  segments: optional [(column end, t column)] pairs
    (at most 4) mapping output column ranges to their adapter's t columns."""
    N, r = B.shape
    if qw.shape[0] != N:
        raise ValueError("B must have one row per output column")
    segs = list(segments) if segments else []
    if len(segs) > 4:
        raise ValueError("at most 4 segments")
    tmax = max([c for _, c in segs], default=0) + lora_pad(r)
    ldt = _lora_t(t, B, tmax, qx.shape[0])
    ends = (C.c_int64 * 4)(*[e for e, _ in segs] + [0] * (4 - len(segs)))
    cols = (C.c_int64 * 4)(*[c for _, c in segs] + [0] * (4 - len(segs)))
    return _w8a8_lora("clef_w8a8_linear_lora", qx, sx, qw, sw, bias, y, N, stream,
                      (_ptr(t), ldt, _ptr(B), r, len(segs), ends, cols))


def w8a8_gateup_swiglu_lora(qx, sx, qw_gu, sw_gu, bias_gu, t_gu, B_gate, B_up, h=None, stream=None):
    """INT8 gate/up SwiGLU with the gate and up LoRA adds fused: the bytes of
    w8a8_linear on the packed weight followed by lora_gateup_swiglu.  t_gu:
    bf16 [M][2 r_pad] = [x A_gate^T | x A_up^T] (one lora_shrink over the
    stacked, padded A factors); B_gate, B_up: bf16 [N][r]."""
    N = _gateup_half(qw_gu)
    r = B_gate.shape[1]
    if B_gate.shape != (N, r) or B_up.shape != (N, r):
        raise ValueError("B_gate and B_up must be [N][r]")
    _cuda(B_up, "B_up", (torch.bfloat16,))
    _dense(B_up, "B_up")
    ldt = _lora_t(t_gu, B_gate, 2 * lora_pad(r), qx.shape[0])
    return _w8a8_lora("clef_w8a8_gateup_swiglu_lora", qx, sx, qw_gu, sw_gu, bias_gu, h, N, stream,
                      (_ptr(t_gu), ldt, _ptr(B_gate), _ptr(B_up), r))


def _w8a8_lora(name, qx, sx, qw, sw, bias, out, n_out, stream, lora_args):
    # the same checks as the plain calls (lengths the C ABI cannot see)
    _w8a8_checks((torch.int8,), qx, sx, qw, sw, bias)
    M, K = qx.shape
    if out is None:
        out = torch.empty((M, n_out), dtype=torch.bfloat16, device=qx.device)
    _cuda(out, "out", (torch.bfloat16,))
    _out_shape(out, M, n_out)
    ldo = _rows(out, "out")
    L = library()
    fn = getattr(L, name)
    rc = fn(_ptr(qx), _ptr(sx), _ptr(qw), _ptr(sw), _ptr(bias), M, n_out, K, *lora_args, _ptr(out), ldo,
            _stream(qx, stream))
    if rc != 0:
        raise ClefError(name, rc, L.clef_last_error().decode(errors="replace"))
    return out


def w8a8_gemm_s32(qx, qw, acc=None, stream=None):
    """Exact int32 accumulators of the INT8 GEMM (same kernel as w8a8_linear)."""
    _cuda(qx, "qx", (torch.int8,)); _cuda(qw, "qw", (torch.int8,))
    _dense(qx, "qx"); _dense(qw, "qw")
    M, K = qx.shape
    N = qw.shape[0]
    if qw.shape[1] != K:
        raise ValueError("qx and qw disagree on K")
    if acc is None:
        acc = torch.empty((M, N), dtype=torch.int32, device=qx.device)
    _cuda(acc, "acc", (torch.int32,))
    _out_shape(acc, M, N)
    _call("clef_w8a8_gemm_s32", _ptr(qx), _ptr(qw), M, N, K, _ptr(acc), _rows(acc, "acc"),
          _stream(qx, stream))
    return acc


_BOUND = {}


def gemm_workspace_bytes() -> int:
    """Bytes of the stream-K workspace on the current device."""
    n = C.c_int64(0)
    _call("clef_gemm_workspace_bytes", C.c_void_p(C.addressof(n)))
    return n.value


def bind_workspace(ws, stream=None):
    """Bind a zero-filled uint8 CUDA buffer of gemm_workspace_bytes() to
    `stream` (default: the current stream) so that INT8 GEMMs and FP8 linears
    launched on it may split tiles across SMs; ws = None unbinds.  The buffer is kept alive
    while bound."""
    s = stream if stream is not None else torch.cuda.current_stream()
    key = (torch.cuda.current_device(), s.cuda_stream)
    if ws is None:
        _call("clef_bind_workspace", C.c_void_p(s.cuda_stream), C.c_void_p(None), 0)
        _BOUND.pop(key, None)
        return
    _cuda(ws, "ws", (torch.uint8,))
    _dense(ws, "ws")
    _call("clef_bind_workspace", C.c_void_p(s.cuda_stream), _ptr(ws), ws.numel())
    _BOUND[key] = ws


def lora_pad(r: int) -> int:
    return (r + 63) // 64 * 64


def lora_add(x, A, B, y, t_scratch=None, stream=None):
    """In place: y = bf16(y + bf16(x A^T) B^T).  Returns y."""
    for t, n in ((x, "x"), (A, "A"), (B, "B"), (y, "y")):
        _cuda(t, n, (torch.bfloat16,))
    _dense(A, "A"); _dense(B, "B")
    M, K = x.shape
    r = A.shape[0]
    N = B.shape[0]
    if A.shape[1] != K or B.shape[1] != r or y.shape != (M, N):
        raise ValueError("LoRA shapes disagree")
    if t_scratch is None:
        t_scratch = torch.empty((M, lora_pad(r)), dtype=torch.bfloat16, device=x.device)
    _dense(t_scratch, "t_scratch")
    _call("clef_lora_add", _ptr(x), _rows(x, "x"), _ptr(A), _ptr(B), M, K, N, r, _ptr(t_scratch),
          _ptr(y), _rows(y, "y"), _stream(x, stream))
    return y


def lora_shrink(x, A, t=None, stream=None):
    """t[:, :lora_pad(r)] = bf16(x A^T), rows of A past r read as zeros.
    A may hold several adapters' factors stacked (each padded to 64 rows);
    t may be a column block of a wider buffer.  Returns t."""
    for a, n in ((x, "x"), (A, "A")):
        _cuda(a, n, (torch.bfloat16,))
    _dense(A, "A")
    M, K = x.shape
    r = A.shape[0]
    if A.shape[1] != K:
        raise ValueError("LoRA shapes disagree")
    if t is None:
        t = torch.empty((M, lora_pad(r)), dtype=torch.bfloat16, device=x.device)
    _cuda(t, "t", (torch.bfloat16,))
    if t.shape[0] != M or t.shape[1] < lora_pad(r):
        raise ValueError("t must have M rows and at least round_up(r, 64) columns")
    _call("clef_lora_shrink", _ptr(x), _rows(x, "x"), _ptr(A), M, K, r, _ptr(t), _rows(t, "t"),
          _stream(x, stream))
    return t


def lora_expand_add(t, B, y, stream=None):
    """In place: y = bf16(y + t[:, :r] B^T) with r = B.shape[1] (t's columns
    r .. lora_pad(r) - 1 must be finite; they meet zeros).  Returns y."""
    for a, n in ((t, "t"), (B, "B"), (y, "y")):
        _cuda(a, n, (torch.bfloat16,))
    _dense(B, "B")
    M = y.shape[0]
    N, r = B.shape
    if t.shape[0] != M or t.shape[1] < lora_pad(r) or y.shape[1] != N:
        raise ValueError("LoRA shapes disagree")
    _call("clef_lora_expand_add", _ptr(t), _rows(t, "t"), _ptr(B), M, N, r, _ptr(y), _rows(y, "y"),
          _stream(y, stream))
    return y


def lora_add_noalloc(x, A, B, y, stream=None):
    """In place: y = bf16(y + bf16(x A^T) B^T), with t kept in the library's
    built-in device scratch (for callers that cannot allocate).  Returns y."""
    for t, n in ((x, "x"), (A, "A"), (B, "B"), (y, "y")):
        _cuda(t, n, (torch.bfloat16,))
    _dense(A, "A"); _dense(B, "B")
    M, K = x.shape
    r = A.shape[0]
    N = B.shape[0]
    if A.shape[1] != K or B.shape[1] != r or y.shape != (M, N):
        raise ValueError("LoRA shapes disagree")
    _call("clef_lora_add_noalloc", _ptr(x), _rows(x, "x"), _ptr(A), _ptr(B), M, K, N, r,
          _ptr(y), _rows(y, "y"), _stream(x, stream))
    return y


def lora_gateup_swiglu(x, A_gate, B_gate, A_up, B_up, y_gu, h=None, t_scratch=None, stream=None):
    """h = bf16(silu(g) * u) with g, u the gate and up halves of y_gu after
    their LoRA adds (each as lora_add computes it).  y_gu is read only."""
    for t, n in ((x, "x"), (A_gate, "A_gate"), (B_gate, "B_gate"), (A_up, "A_up"), (B_up, "B_up"),
                 (y_gu, "y_gu")):
        _cuda(t, n, (torch.bfloat16,))
    for t, n in ((A_gate, "A_gate"), (B_gate, "B_gate"), (A_up, "A_up"), (B_up, "B_up")):
        _dense(t, n)
    M, K = x.shape
    r = A_gate.shape[0]
    N = B_gate.shape[0]
    if (A_gate.shape != (r, K) or A_up.shape != (r, K) or B_gate.shape != (N, r) or B_up.shape != (N, r)
            or y_gu.shape != (M, 2 * N)):
        raise ValueError("LoRA gate/up shapes disagree")
    if t_scratch is None:
        t_scratch = torch.empty((M, 2 * lora_pad(r)), dtype=torch.bfloat16, device=x.device)
    _dense(t_scratch, "t_scratch")
    if h is None:
        h = torch.empty((M, N), dtype=torch.bfloat16, device=x.device)
    _cuda(h, "h", (torch.bfloat16,))
    _call("clef_lora_gateup_swiglu", _ptr(x), _rows(x, "x"), _ptr(A_gate), _ptr(B_gate), _ptr(A_up),
          _ptr(B_up), M, K, N, r, _ptr(t_scratch), _ptr(y_gu), _rows(y_gu, "y_gu"), _ptr(h), _rows(h, "h"),
          _stream(x, stream))
    return h


def swiglu_bf16(y_gu, h=None, stream=None):
    """Unfused MLP product: h = bf16(silu(g) * u) of bf16 [M][2N] gate|up rows."""
    _cuda(y_gu, "y_gu", (torch.bfloat16,))
    M, N2 = y_gu.shape
    N = N2 // 2
    if h is None:
        h = torch.empty((M, N), dtype=torch.bfloat16, device=y_gu.device)
    _call("clef_swiglu_bf16", _ptr(y_gu), M, N, _rows(y_gu, "y_gu"), _ptr(h), _rows(h, "h"),
          _stream(y_gu, stream))
    return h


MMA_KINDS = {"bf16": 0, "e4m3": 1, "s8_mma_sync": 2}


def mma_peak(kind: str, iters: int = 200_000) -> float:
    """Dense tensor-core rate (TFLOP/s) of one instruction route on the
    current device, from the library's microbenchmark: "bf16" (tcgen05
    kind::f16), "e4m3" (tcgen05 kind::f8f6f4) or "s8_mma_sync"."""
    out = C.c_double(0.0)
    _call("clef_mma_peak", MMA_KINDS[kind], int(iters), C.c_void_p(C.addressof(out)))
    return out.value


def poll_status() -> int:
    """Synchronise and return (then clear) the device-side status word."""
    return int(library().clef_poll_status())


def set_wait_limit_ns(ns: int) -> None:
    library().clef_set_wait_limit_ns(int(ns))


def set_quant_staging(mode: int) -> None:
    """Choose the quantizer kernel: 1 (default) the TMA-staged persistent one
    for large calls, 2 the staged one wherever the row length suits it, 0
    always the one-CTA-per-row kernel."""
    L = library()
    L.clef_set_quant_staging.argtypes = [C.c_int]
    L.clef_set_quant_staging.restype = None
    L.clef_set_quant_staging(int(mode))


def set_pdl(on: bool) -> None:
    """Programmatic dependent launch for later launches (default on): a
    kernel may start its set-up while the stream's previous kernel finishes;
    the bytes computed are the same either way."""
    L = library()
    L.clef_set_pdl.argtypes = [C.c_int]
    L.clef_set_pdl.restype = None
    L.clef_set_pdl(1 if on else 0)


def set_sm_budget(sms: int) -> None:
    """SMs the library's later compute launches may fill (0: all of them;
    rounded down to an even count).  The bytes computed do not depend on it;
    SMs outside the budget stay free for work on other streams, such as
    copy_sm moving the next step's inputs."""
    _call("clef_set_sm_budget", int(sms))


def copy_sm(dst: torch.Tensor, src: torch.Tensor, ctas: int = 4, stream=None) -> torch.Tensor:
    """Copy src into dst (same byte count, both contiguous) with loads and
    stores issued by `ctas` CTAs instead of a copy engine.  Each side is a
    CUDA tensor or a page-locked CPU tensor.  Returns dst."""
    for t, n in ((dst, "dst"), (src, "src")):
        if not isinstance(t, torch.Tensor):
            raise ValueError(f"{n} must be a tensor")
        _dense(t, n)
        if not t.is_cuda and not t.is_pinned():
            raise ValueError(f"{n} must be a CUDA tensor or a page-locked CPU tensor")
    nbytes = dst.numel() * dst.element_size()
    if src.numel() * src.element_size() != nbytes:
        raise ValueError("dst and src differ in size")
    dev = dst if dst.is_cuda else src
    if not dev.is_cuda:
        raise ValueError("one side must be a CUDA tensor (its device runs the copy)")
    _call("clef_copy_sm", _ptr(dst), _ptr(src), nbytes, int(ctas), _stream(dev, stream))
    return dst


def test_force_timeout(on) -> None:
    """Test knob: make the GEMM kernels' MMA issuer wait on a barrier nothing
    signals.  True / 1: every CTA; an int n >= 2: only the CTA (pair) of
    tile-loop slot n - 2; False / 0: off."""
    L = library()
    L.clef_test_force_timeout.argtypes = [C.c_int]
    L.clef_test_force_timeout.restype = None
    L.clef_test_force_timeout(int(on) if not isinstance(on, bool) else (1 if on else 0))
