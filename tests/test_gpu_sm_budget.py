"""clef_copy_sm (a copy issued by a few CTAs instead of a copy engine) and
clef_set_sm_budget (the SMs the compute launches may fill).

The copy must move every byte between device memory and page-locked host
memory in both directions and within the device, for sizes that are not a
multiple of the CTAs' stride and any CTA count.  Compute launches under any
budget must give the bytes of the unrestricted launches: the tile order and
every split follow the shapes, only the number of persistent CTAs changes
(INT8 stream-K pieces, FP8 K parts, the quantizer's two kernels, the fused
LoRA and a whole layer step).  A copy running on a side stream beside a GEMM
under a budget that leaves it room must leave both results intact."""
import ctypes as C

import numpy as np
import pytest
import torch

import clef_synth as S
import w8a8_quantized_projections_gb300 as clef
from clef_synth.configs import Config, Projection
from gpu_util import bf16_dev, bf16_host
from w8a8_quantized_projections_gb300.layer import QuantizedLayer

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    yield
    clef.set_sm_budget(0)
    assert clef.poll_status() == 0


def _bytes(n, seed):
    g = torch.Generator().manual_seed(seed)
    return torch.randint(-128, 128, (n,), dtype=torch.int8, generator=g)


@pytest.mark.parametrize("n", [16, 4096 + 16, (1 << 20) + 48, 3 * (1 << 24) + 1024 * 16 * 8 + 16])
@pytest.mark.parametrize("ctas", [1, 3, 4, 8])
def test_copy_directions(n, ctas):
    src_h = _bytes(n, n + ctas).pin_memory()
    dev = torch.empty(n, dtype=torch.int8, device="cuda")
    clef.copy_sm(dev, src_h, ctas)                        # host -> device
    dev2 = torch.empty_like(dev)
    clef.copy_sm(dev2, dev, ctas)                         # device -> device
    back = torch.empty(n, dtype=torch.int8).pin_memory()
    clef.copy_sm(back, dev2, ctas)                        # device -> host
    torch.cuda.synchronize()
    assert torch.equal(dev.cpu(), src_h)
    assert torch.equal(back, src_h)


def test_copy_from_pageable_host_memory_is_refused_or_correct():
    """Through the C ABI, pageable host memory (a numpy buffer) is either
    refused on the host (nothing launched) or, where the device reads
    pageable memory directly, copied byte for byte."""
    n = (1 << 20) + 16
    src = np.random.default_rng(5).integers(-128, 128, n, dtype=np.int8)
    assert src.ctypes.data % 16 == 0
    dst = torch.zeros(n, dtype=torch.int8, device="cuda")
    rc = clef.library().clef_copy_sm(C.c_void_p(dst.data_ptr()), C.c_void_p(src.ctypes.data), n, 4,
                                     C.c_void_p(torch.cuda.current_stream().cuda_stream))
    torch.cuda.synchronize()
    assert rc in (0, 1)
    if rc == 0:
        assert np.array_equal(dst.cpu().numpy(), src)
    else:
        assert b"page-locked" in clef.library().clef_last_error()
        assert int(dst.count_nonzero()) == 0


def test_copy_refuses_unpinned_and_mismatched():
    dev = torch.empty(64, dtype=torch.int8, device="cuda")
    with pytest.raises(ValueError, match="page-locked"):
        clef.copy_sm(dev, torch.zeros(64, dtype=torch.int8))
    with pytest.raises(ValueError, match="size"):
        clef.copy_sm(dev, torch.zeros(80, dtype=torch.int8).pin_memory())


def _eq(a, b, what):
    assert torch.equal(a.view(torch.int16), b.view(torch.int16)), what


def _codes(tag, M, N, K, mode="int8_h128"):
    x = bf16_dev(S.activation(0, f"t/smb/{tag}/x", M, K))
    w = bf16_dev(S.weight(0, f"t/smb/{tag}/w", N, K))
    b = bf16_dev(S.bias(0, f"t/smb/{tag}/b", N))
    return x, w, b


BUDGETS = [148, 100, 2]


def test_linear_and_quantizer_under_budgets():
    """INT8 linear with stream-K (a workspace bound; 1,502 x 5120 x 17408
    leaves a partial last wave), FP8 linear with K parts (K = 8192), the
    quantizer (staged and per-row kernels are chosen by rows per SM)."""
    ws = torch.zeros(clef.gemm_workspace_bytes(), dtype=torch.uint8, device="cuda")
    clef.bind_workspace(ws)
    x, w, b = _codes("i8", 1502, 5120, 17408)
    xf, wf, bf = _codes("f8", 1502, 4096, 8192)

    def run():
        qx, sx = clef.quant_act(x, "int8_h128")
        qw, sw = clef.quant_act(w, "int8_h128")
        y = clef.w8a8_linear(qx, sx, qw, sw, b)
        fx, fsx = clef.quant_act(xf, "fp8")
        fw, fsw = clef.quant_act(wf, "fp8")
        yf = clef.fp8_linear(fx, fsx, fw, fsw, bf)
        return qx, sx, y, yf

    try:
        ref = run()
        for budget in BUDGETS:
            clef.set_sm_budget(budget)
            got = run()
            torch.cuda.synchronize()
            assert torch.equal(got[0], ref[0]) and torch.equal(got[1], ref[1]), budget
            _eq(got[2], ref[2], f"int8 linear, budget {budget}")
            _eq(got[3], ref[3], f"fp8 linear, budget {budget}")
    finally:
        torch.cuda.synchronize()
        clef.bind_workspace(None)
        clef.set_sm_budget(0)


def test_layer_step_under_budgets():
    proj = [Projection("q", 1024, 1024, act="x_attn"), Projection("k", 1024, 256, act="x_attn"),
            Projection("v", 1024, 256, act="x_attn"), Projection("o", 1024, 1024, act="x_o"),
            Projection("gateup", 1024, 2048, kind="gateup", act="x_mlp"),
            Projection("down", 2048, 1024, act="x_down", chained=True)]
    cfg = Config(93, "smb-layer", 1502, "int8", proj, lora_rank=64)
    acts_np, weights_np, lora_np = S.layer_inputs(cfg, seed=7)
    weights = {k: (bf16_dev(W), bf16_dev(bb)) for k, (W, bb) in weights_np.items()}
    lora = {k: (bf16_dev(A), bf16_dev(B)) for k, (A, B) in lora_np.items()}
    acts = {k: bf16_dev(v) for k, v in acts_np.items()}
    layer = QuantizedLayer(cfg, weights, lora)
    ref = {k: bf16_host(v) for k, v in layer.step(acts).items()}
    for budget in BUDGETS:
        clef.set_sm_budget(budget)
        out = {k: bf16_host(v) for k, v in layer.step(acts).items()}
        for k in ref:
            assert np.array_equal(out[k], ref[k]), (budget, k)
    clef.set_sm_budget(0)


def test_copy_beside_gemm():
    """A copy of 256 MB on a side stream while a GEMM runs on the main
    stream, the compute under a budget of every SM but the copy's four."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    x, w, b = _codes("beside", 4096, 8192, 5120)
    qx, sx = clef.quant_act(x, "int8_h128")
    qw, sw = clef.quant_act(w, "int8_h128")
    ref = clef.w8a8_linear(qx, sx, qw, sw, b)
    src = _bytes(256 << 20, 3).pin_memory()
    dst = torch.empty(src.numel(), dtype=torch.int8, device="cuda")
    side = torch.cuda.Stream()
    clef.set_sm_budget(sms - 4)
    torch.cuda.synchronize()
    with torch.cuda.stream(side):
        clef.copy_sm(dst, src, 4, stream=side)
    ys = [clef.w8a8_linear(qx, sx, qw, sw, b) for _ in range(3)]
    torch.cuda.synchronize()
    clef.set_sm_budget(0)
    for y in ys:
        _eq(y, ref, "GEMM beside the copy")
    assert torch.equal(dst.cpu(), src)
