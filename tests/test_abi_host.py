"""Host-side checks of the C ABI that need no GPU: the library builds for
sm_103a, loads, exports every function include/clef.h declares, and rejects
bad arguments on the host before touching any device (no compute call)."""
import ctypes as C
import os
import re

import pytest

import w8a8_quantized_projections_gb300 as clef

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    src = open(os.path.join(ROOT, "include", "clef.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(clef_[a-z0-9_]+)\s*\(", src)))


def test_library_exports_every_declared_symbol():
    L = clef.library()
    names = declared_functions()
    assert len(names) >= 12
    for n in names:
        assert hasattr(L, n), n


def test_status_strings_and_version():
    L = clef.library()
    assert L.clef_status_string(0) == b"CLEF_OK"
    assert L.clef_status_string(4) == b"CLEF_ERR_TIMEOUT"
    assert L.clef_abi_version() == 100


FAKE = C.c_void_p(0x10000)       # 16-byte aligned, never dereferenced
ODD = C.c_void_p(0x10008)        # 8-byte aligned only
NUL = C.c_void_p(None)
S = C.c_void_p(None)             # stream


@pytest.mark.parametrize("args", [
    (NUL, 4, 128, 128, 0, FAKE, FAKE, S),       # null x
    (FAKE, 4, 100, 128, 0, FAKE, FAKE, S),      # K not a multiple of 128 (rotated)
    (FAKE, 4, 80, 80, 1, FAKE, FAKE, S),        # K not a multiple of 32 (fp8)
    (FAKE, 4, 96, 96, 2, FAKE, FAKE, S),        # K not a multiple of 128 (rotated fp8)
    (FAKE, 4, 128, 120, 0, FAKE, FAKE, S),      # ldx < K
    (ODD, 4, 128, 128, 0, FAKE, FAKE, S),       # misaligned x
    (FAKE, 4, 128, 128, 7, FAKE, FAKE, S),      # unknown mode
    (FAKE, -1, 128, 128, 0, FAKE, FAKE, S),     # negative M
    (FAKE, 4, 131072, 131072, 0, FAKE, FAKE, S),  # K too large
])
def test_quant_act_rejects_bad_arguments(args):
    assert clef.library().clef_quant_act(*args) == 1


@pytest.mark.parametrize("sc", [0.0, -1.0, float("inf"), float("nan")])
def test_quant_act_static_rejects_bad_scales(sc):
    assert clef.library().clef_quant_act_static(FAKE, 4, 128, 128, 1, sc, FAKE, FAKE, S) == 1


@pytest.mark.parametrize("mode", [0, 2])
def test_quant_act_static_rotated_needs_whole_blocks(mode):
    assert clef.library().clef_quant_act_static(FAKE, 4, 96, 96, mode, 0.5, FAKE, FAKE, S) == 1


@pytest.mark.parametrize("name", ["clef_w8a8_linear", "clef_fp8_linear", "clef_w8a8_gateup_swiglu",
                                  "clef_fp8_gateup_swiglu"])
@pytest.mark.parametrize("bad", ["null_qx", "N8", "K16", "ldy", "align", "sw_align", "bias_align"])
def test_gemm_rejects_bad_arguments(name, bad):
    qx, sx, qw, sw, bias, M, N, K, y, ldy = FAKE, FAKE, FAKE, FAKE, NUL, 4, 256, 256, FAKE, 256
    if bad == "null_qx":
        qx = NUL
    elif bad == "N8":
        N, ldy = 20, 20
    elif bad == "K16":
        K = 40
    elif bad == "ldy":
        ldy = 100
    elif bad == "align":
        y = ODD
    elif bad == "sw_align":
        sw = ODD
    elif bad == "bias_align":     # the epilogue reads 8 bias columns per 16-byte load
        bias = ODD
    assert getattr(clef.library(), name)(qx, sx, qw, sw, bias, M, N, K, y, ldy, S) == 1


@pytest.mark.parametrize("bad", ["rank", "rank8", "K", "ldy", "null_t"])
def test_lora_rejects_bad_arguments(bad):
    x, ldx, A, B, M, K, N, r, t, y, ldy = FAKE, 256, FAKE, FAKE, 4, 256, 64, 48, FAKE, FAKE, 64
    if bad == "rank":
        r = 0
    elif bad == "rank8":
        r = 50
    elif bad == "K":
        K = 12
    elif bad == "ldy":
        ldy = 60
    elif bad == "null_t":
        t = NUL
    assert clef.library().clef_lora_add(x, ldx, A, B, M, K, N, r, t, y, ldy, S) == 1


@pytest.mark.parametrize("bad", ["rank", "rank_big", "K", "ldx", "ldt", "ldt8", "null_x", "align_t"])
def test_lora_shrink_rejects_bad_arguments(bad):
    x, ldx, A, M, K, r, t, ldt = FAKE, 256, FAKE, 4, 256, 48, FAKE, 64
    if bad == "rank":
        r = 0
    elif bad == "rank_big":
        r = 4104
    elif bad == "K":
        K = 12
    elif bad == "ldx":
        ldx = 128
    elif bad == "ldt":
        ldt = 56       # below round_up(48, 64)
    elif bad == "ldt8":
        ldt = 68
    elif bad == "null_x":
        x = NUL
    elif bad == "align_t":
        t = ODD
    assert clef.library().clef_lora_shrink(x, ldx, A, M, K, r, t, ldt, S) == 1


@pytest.mark.parametrize("bad", ["rank", "N", "ldt", "ldy", "null_B", "align_y"])
def test_lora_expand_add_rejects_bad_arguments(bad):
    t, ldt, B, M, N, r, y, ldy = FAKE, 64, FAKE, 4, 64, 48, FAKE, 64
    if bad == "rank":
        r = 12
    elif bad == "N":
        N = 60
    elif bad == "ldt":
        ldt = 48       # below round_up(48, 64)
    elif bad == "ldy":
        ldy = 32
    elif bad == "null_B":
        B = NUL
    elif bad == "align_y":
        y = ODD
    assert clef.library().clef_lora_expand_add(t, ldt, B, M, N, r, y, ldy, S) == 1


@pytest.mark.parametrize("bad", ["align", "small"])
def test_bind_workspace_rejects_bad_arguments(bad):
    ws, n = FAKE, 1 << 26
    if bad == "align":
        ws = ODD
    else:
        n = 1024           # below the counter block
    assert clef.library().clef_bind_workspace(S, ws, n) == 1


def test_workspace_bytes_rejects_null():
    assert clef.library().clef_gemm_workspace_bytes(NUL) == 1


def test_valid_arguments_without_gpu_report_device_error():
    """With valid arguments the call reaches the device checks; on a machine
    without a usable sm_103 GPU that is an error code, never a crash."""
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    rc = clef.library().clef_quant_act(FAKE, 4, 128, 128, 0, FAKE, FAKE, S)
    assert rc in (2, 3)


def test_python_binding_rejects_cpu_tensors():
    import torch
    with pytest.raises(ValueError):
        clef.quant_act(torch.zeros(4, 128, dtype=torch.bfloat16))


@pytest.mark.parametrize("kind,iters,out", [(3, 10, True), (-1, 10, True), (0, 0, True), (1, 1 << 25, True),
                                            (0, 10, False)])
def test_mma_peak_rejects_bad_arguments(kind, iters, out):
    d = C.c_double(0.0)
    ptr = C.c_void_p(C.addressof(d)) if out else NUL
    assert clef.library().clef_mma_peak(kind, iters, ptr) == 1


@pytest.mark.parametrize("args", [
    (NUL, FAKE, 64, 4, S),            # null dst
    (FAKE, NUL, 64, 4, S),            # null src
    (ODD, C.c_void_p(0x20000), 64, 4, S),   # misaligned dst
    (FAKE, C.c_void_p(0x20000), 40, 4, S),  # bytes not a multiple of 16
    (FAKE, C.c_void_p(0x20000), -16, 4, S),  # negative
    (FAKE, C.c_void_p(0x20000), 64, 0, S),   # no CTA
    (FAKE, C.c_void_p(0x20000), 64, 65, S),  # too many CTAs
    (FAKE, C.c_void_p(0x10010), 64, 4, S),   # overlapping ranges
])
def test_copy_sm_rejects_bad_arguments(args):
    assert clef.library().clef_copy_sm(*args) == 1


def test_copy_sm_empty_is_ok_without_launch():
    assert clef.library().clef_copy_sm(NUL, NUL, 0, 4, S) == 0


def test_sm_budget_arguments():
    L = clef.library()
    assert L.clef_set_sm_budget(-1) == 1
    assert L.clef_set_sm_budget(1) == 1
    assert L.clef_set_sm_budget(148) == 0
    assert L.clef_set_sm_budget(0) == 0
