"""The binding's checks of buffer lengths the C ABI cannot see (it receives
bare pointers): short or long scale and bias vectors, an odd packed gate/up
row count and an output of the wrong shape are refused before any launch."""
import pytest
import torch

import w8a8_quantized_projections_gb300 as clef

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def _codes(M, N, K):
    qx = torch.zeros((M, K), dtype=torch.int8, device="cuda")
    qw = torch.zeros((N, K), dtype=torch.int8, device="cuda")
    return qx, qw


@pytest.mark.parametrize("fn", ["w8a8_linear", "fp8_linear"])
def test_scale_and_bias_lengths(fn):
    M, N, K = 64, 128, 256
    qx, qw = _codes(M, N, K)
    if fn == "fp8_linear":
        qx, qw = qx.view(torch.uint8), qw.view(torch.uint8)
    f = getattr(clef, fn)
    sx = torch.ones(M, device="cuda")
    sw = torch.ones(N, device="cuda")
    bias = torch.zeros(N, dtype=torch.bfloat16, device="cuda")
    f(qx, sx, qw, sw, bias)                      # the right lengths pass
    with pytest.raises(ValueError, match="sx"):
        f(qx, sx[:-1], qw, sw, bias)
    with pytest.raises(ValueError, match="sw"):
        f(qx, sx, qw, sw[:-8], bias)
    with pytest.raises(ValueError, match="bias"):
        f(qx, sx, qw, sw, bias[:-8])
    with pytest.raises(ValueError, match="bias"):
        f(qx, sx, qw, sw, torch.zeros(N + 8, dtype=torch.bfloat16, device="cuda"))
    torch.cuda.synchronize()
    assert clef.poll_status() == 0


@pytest.mark.parametrize("fn", ["w8a8_gateup_swiglu", "fp8_gateup_swiglu"])
def test_gateup_rows_even_and_lengths(fn):
    M, K = 64, 256
    qx, qw = _codes(M, 2 * 128, K)
    if fn.startswith("fp8"):
        qx, qw = qx.view(torch.uint8), qw.view(torch.uint8)
    f = getattr(clef, fn)
    sx = torch.ones(M, device="cuda")
    sw = torch.ones(256, device="cuda")
    f(qx, sx, qw, sw)
    with pytest.raises(ValueError, match="even"):
        f(qx, sx, qw[:-1], sw[:-1])
    with pytest.raises(ValueError, match="sw"):
        f(qx, sx, qw, sw[:128])
    torch.cuda.synchronize()
    assert clef.poll_status() == 0


def test_output_shape():
    M, N, K = 64, 128, 256
    qx, qw = _codes(M, N, K)
    sx = torch.ones(M, device="cuda")
    sw = torch.ones(N, device="cuda")
    wide = torch.zeros((M, N + 8), dtype=torch.bfloat16, device="cuda")
    clef.w8a8_linear(qx, sx, qw, sw, y=wide[:, :N])          # a window of the right shape passes
    for bad in (wide[:, :N - 8], wide[:M - 1, :N], wide):
        with pytest.raises(ValueError, match="shape"):
            clef.w8a8_linear(qx, sx, qw, sw, y=bad)
    with pytest.raises(ValueError, match="shape"):
        clef.w8a8_gateup_swiglu(qx, sx, qw, sw, h=wide[:, :N])   # h has N / 2 columns
    t = torch.zeros((M, 64), dtype=torch.bfloat16, device="cuda")
    B = torch.zeros((N, 64), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(ValueError, match="shape"):
        clef.w8a8_linear_lora(qx, sx, qw, sw, None, t, B, y=wide[:, :N - 8])
    with pytest.raises(ValueError, match="shape"):
        clef.w8a8_gemm_s32(qx, qw, acc=torch.zeros((M, N - 8), dtype=torch.int32, device="cuda"))
    torch.cuda.synchronize()
    assert clef.poll_status() == 0
