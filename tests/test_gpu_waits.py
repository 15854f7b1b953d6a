"""Device-side failure handling without a GPU fault.

Every wait inside the GEMM kernels is time-limited.  With the test knob on,
the MMA issuer waits on a barrier that nothing signals; after the time limit
(2 ms here) the kernel records CLEF_ERR_TIMEOUT in the library's status word,
lets the copies it already issued land, frees its tensor memory and returns.  The test checks the
status is reported, then restores the limit and checks that the same CUDA
context still computes bit-exact results (single-CTA and CTA-pair tiles, INT8
and FP8)."""
import numpy as np
import pytest
import torch

import clef_synth as S
import w8a8_quantized_projections_gb300 as clef
from gpu_util import bf16_dev, bf16_host, host

pytestmark = pytest.mark.gpu

TIMEOUT = 4


@pytest.fixture(autouse=True)
def _restore_limit():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    yield
    clef.test_force_timeout(False)
    clef.set_wait_limit_ns(10 ** 9)


@pytest.mark.parametrize("M", [64, 512])
def test_timeout_reported_and_context_survives(orc, M):
    N, K = 512, 2048
    x = S.activation(0, f"t/wait/x{M}", M, K)
    w = S.weight(0, "t/wait/w", N, K)
    qx, sx = clef.quant_act(bf16_dev(x), "int8_h128")
    qw, sw = clef.quant_act(bf16_dev(w), "int8_h128")
    fx, fsx = clef.quant_act(bf16_dev(x), "fp8")
    fw, fsw = clef.quant_act(bf16_dev(w), "fp8")
    assert clef.poll_status() == 0

    clef.set_wait_limit_ns(2_000_000)
    clef.test_force_timeout(True)
    clef.w8a8_linear(qx, sx, qw, sw)
    assert clef.poll_status() == TIMEOUT
    clef.fp8_linear(fx, fsx, fw, fsw)
    assert clef.poll_status() == TIMEOUT
    clef.test_force_timeout(False)
    clef.set_wait_limit_ns(10 ** 9)

    y = bf16_host(clef.w8a8_linear(qx, sx, qw, sw))
    ref = orc.int8_linear(host(qx), host(sx), host(qw), host(sw))
    assert np.array_equal(y, ref)
    assert clef.poll_status() == 0


def test_split_launch_timeout_then_layer_refill():
    """Only one CTA pair of a stream-K launch gives up (the knob on tile-loop
    slot 0): the other pairs finish, and the arrival counters of the split
    tiles slot 0 shared stay nonzero in the workspace.  QuantizedLayer's
    poll_status reports the time-out and refills the workspace with zeros;
    the next step is then byte-equal to a clean one."""
    from clef_synth.configs import Config, Projection
    from w8a8_quantized_projections_gb300.layer import QuantizedLayer

    # 1502 x 5120 x 17408: 120 tiles on 76 CTA pairs, the last 44 split
    cfg = Config(90, "wait-test-down-m1502", 1502, "int8", [Projection("down", 17408, 5120, act="x")])
    x = bf16_dev(S.activation(0, "t/wait/split/x", cfg.M, 17408))
    W = bf16_dev(S.weight(0, "t/wait/split/w", 5120, 17408))
    b = bf16_dev(S.bias(0, "t/wait/split/b", 5120))
    layer = QuantizedLayer(cfg, {"down": (W, b)})
    ref = bf16_host(layer.step({"x": x})["down"])
    assert layer.poll_status() == 0

    clef.set_wait_limit_ns(20_000_000)
    clef.test_force_timeout(2)        # slot 0 only
    layer.step({"x": x})
    torch.cuda.synchronize()
    clef.test_force_timeout(False)
    counters = layer.ws[: 4096 * 2 * 8 * 4].view(torch.int32)
    assert int((counters != 0).sum()) > 0, "the aborted pair left arrival counts behind"
    assert layer.poll_status() == TIMEOUT
    assert int((counters != 0).sum()) == 0, "workspace refilled"
    clef.set_wait_limit_ns(10 ** 9)

    got = bf16_host(layer.step({"x": x})["down"])
    assert np.array_equal(got, ref)
    assert layer.poll_status() == 0
