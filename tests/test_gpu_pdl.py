"""Programmatic dependent launch: a layer step whose launches may overlap
their set-up with the previous kernel's tail computes the same bytes as the
step in plain stream order, over many back-to-back steps (INT8 with LoRA
fused and unfused, FP8; per-row and staged quantizer; stream-K splits)."""
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
def _pdl_default():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    yield
    clef.set_pdl(True)
    clef.set_quant_staging(1)
    assert clef.poll_status() == 0


def layer_cfg(scheme, M, lora_rank):
    proj = [Projection("q", 1024, 1024, act="x_attn"), Projection("k", 1024, 256, act="x_attn"),
            Projection("v", 1024, 256, act="x_attn"), Projection("o", 1024, 1024, act="x_o"),
            Projection("gateup", 1024, 2048, kind="gateup", act="x_mlp"),
            Projection("down", 2048, 1024, act="x_down", chained=True)]
    return Config(91, f"pdl-{scheme}-{M}", M, scheme, proj, lora_rank=lora_rank)


@pytest.mark.parametrize("scheme,M,lora_rank,fuse,staging", [
    ("int8", 300, 64, True, 1),      # per-row quantizer, fused LoRA
    ("int8", 1502, 64, False, 1),    # staged quantizer, unfused LoRA launches, stream-K down
    ("int8", 1502, None, True, 0),   # per-row quantizer on a staged-size call
    ("fp8", 1502, None, True, 1),
])
def test_pdl_steps_equal_plain_order(scheme, M, lora_rank, fuse, staging):
    cfg = layer_cfg(scheme, M, lora_rank)
    acts_np, weights_np, lora_np = S.layer_inputs(cfg, seed=5)
    weights = {k: (bf16_dev(W), bf16_dev(b)) for k, (W, b) in weights_np.items()}
    lora = {k: (bf16_dev(A), bf16_dev(B)) for k, (A, B) in lora_np.items()}
    acts = {k: bf16_dev(x) for k, x in acts_np.items()}
    layer = QuantizedLayer(cfg, weights, lora or None, fuse_lora=fuse)
    clef.set_quant_staging(staging)

    clef.set_pdl(False)
    ref = {k: bf16_host(v) for k, v in layer.step(acts).items()}
    torch.cuda.synchronize()

    clef.set_pdl(True)
    steps = 12
    outs = []
    for _ in range(steps):
        # each step's outputs copied out on the stream, after the step's kernels
        outs.append({k: v.clone() for k, v in layer.step(acts).items()})
    torch.cuda.synchronize()
    for i, o in enumerate(outs):
        for k in ref:
            assert np.array_equal(ref[k], bf16_host(o[k])), (i, k)
