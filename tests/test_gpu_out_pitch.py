"""Outputs at every legal pitch and base.  The GEMM epilogues store a row 16
columns (32 bytes) at a time only where every output row starts on a 32-byte
boundary, and 8 columns at a time elsewhere and past the last whole group of
16 columns.  A call writing into a column window of a wider buffer must give
the bytes of the same call with a dense output, and leave every byte outside
the window as it was: windows with 32-byte rows (wide stores, then a tail of
8 columns when N % 16 == 8), with a pitch of 8 modulo 16 elements, and
starting 8 columns into the buffer (16-byte rows only).  Pair (M > 128) and
single-CTA launches, INT8 and FP8, the scale/bias, SwiGLU and fused LoRA
epilogues, and the LoRA shrink's bf16 store."""
import pytest
import torch

import clef_synth as S
import w8a8_quantized_projections_gb300 as clef
from gpu_util import bf16_dev

pytestmark = pytest.mark.gpu

SENTINEL = -12345   # int16 pattern of the bytes around the window


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    yield
    assert clef.poll_status() == 0


def layouts(N):
    """(row pitch, first column) of the windows: 32-byte rows; a pitch of 8
    modulo 16 elements; a base 8 columns (16 bytes) in."""
    wide = (N + 15) // 16 * 16
    return [(wide if wide > N else N + 16, 0), (wide + 8, 0), (wide + 16, 8)]


def run_windows(call, M, N):
    """call(out) writes the [M][N] output into out (None: a dense output it
    allocates) and returns it."""
    ref = call(None).view(torch.int16)
    for pitch, c0 in layouts(N):
        buf = torch.full((M, pitch), SENTINEL, dtype=torch.int16, device="cuda")
        win = buf.view(torch.bfloat16)[:, c0:c0 + N]
        call(win)
        torch.cuda.synchronize()
        assert torch.equal(buf[:, c0:c0 + N], ref), f"pitch {pitch}, column {c0}"
        outside = torch.cat([buf[:, :c0], buf[:, c0 + N:]], 1)
        assert bool((outside == SENTINEL).all()), f"pitch {pitch}, column {c0}: bytes outside written"


def codes(tag, M, N, K, mode="int8_h128"):
    x = bf16_dev(S.activation(0, f"t/op/{tag}/x", M, K))
    w = bf16_dev(S.weight(0, f"t/op/{tag}/w", N, K))
    b = bf16_dev(S.bias(0, f"t/op/{tag}/b", N))
    qx, sx = clef.quant_act(x, mode)
    qw, sw = clef.quant_act(w, mode)
    return x, qx, sx, qw, sw, b


@pytest.mark.parametrize("M", [300, 100])
@pytest.mark.parametrize("N", [264, 512])
def test_int8_linear(M, N):
    _, qx, sx, qw, sw, b = codes(f"i8lin{M}x{N}", M, N, 1024)
    run_windows(lambda y: clef.w8a8_linear(qx, sx, qw, sw, b, y=y), M, N)


@pytest.mark.parametrize("M", [300, 100])
def test_int8_gateup_swiglu(M):
    N = 136
    _, qx, sx, qw, sw, b = codes(f"i8gu{M}", M, 2 * N, 1024)
    run_windows(lambda h: clef.w8a8_gateup_swiglu(qx, sx, qw, sw, b, h=h), M, N)


@pytest.mark.parametrize("M,K", [(300, 1024), (300, 8192), (100, 1024)])
def test_fp8_linear(M, K):
    """K = 8192 sums each tile's K as three parts before the epilogue."""
    N = 264
    _, qx, sx, qw, sw, b = codes(f"f8lin{M}x{K}", M, N, K, "fp8")
    run_windows(lambda y: clef.fp8_linear(qx, sx, qw, sw, b, y=y), M, N)


@pytest.mark.parametrize("M", [300, 100])
def test_fp8_gateup_swiglu(M):
    N = 136
    _, qx, sx, qw, sw, b = codes(f"f8gu{M}", M, 2 * N, 1024, "fp8")
    run_windows(lambda h: clef.fp8_gateup_swiglu(qx, sx, qw, sw, b, h=h), M, N)


@pytest.mark.parametrize("M", [300, 100])
def test_int8_linear_lora(M):
    N, K, r = 264, 1024, 48
    x, qx, sx, qw, sw, b = codes(f"i8lora{M}", M, N, K)
    A, B = (bf16_dev(v) for v in S.lora_pair(0, f"t/op/i8lora{M}/l", r, K, N))
    t = clef.lora_shrink(x, A)
    run_windows(lambda y: clef.w8a8_linear_lora(qx, sx, qw, sw, b, t, B, y=y), M, N)


@pytest.mark.parametrize("M", [300, 100])
def test_int8_gateup_swiglu_lora(M):
    N, K, r = 136, 1024, 48
    x, qx, sx, qw, sw, b = codes(f"i8gulora{M}", M, 2 * N, K)
    Ag, Bg = (bf16_dev(v) for v in S.lora_pair(0, f"t/op/i8gulora{M}/g", r, K, N))
    Au, Bu = (bf16_dev(v) for v in S.lora_pair(0, f"t/op/i8gulora{M}/u", r, K, N))
    rp = clef.lora_pad(r)
    A = torch.zeros((2 * rp, K), dtype=torch.bfloat16, device="cuda")
    A[:r] = Ag
    A[rp:rp + r] = Au
    t = clef.lora_shrink(x, A)
    run_windows(lambda h: clef.w8a8_gateup_swiglu_lora(qx, sx, qw, sw, b, t, Bg, Bu, h=h), M, N)


@pytest.mark.parametrize("M", [300, 100])
def test_lora_shrink_t(M):
    K, r = 2048, 64
    x = bf16_dev(S.activation(0, f"t/op/shrink{M}/x", M, K))
    A, _ = (bf16_dev(v) for v in S.lora_pair(0, f"t/op/shrink{M}/l", r, K, 64))
    run_windows(lambda t: clef.lora_shrink(x, A, t=t), M, clef.lora_pad(r))
