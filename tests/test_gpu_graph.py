"""A layer step captured in a CUDA graph: its replay reproduces the eager
step's outputs bit for bit (INT8 with q|k|v packing and LoRA adapters, and
FP8), and it recomputes them from the inputs (outputs cleared before the
replay come back; changed inputs give the eager step's new outputs)."""
import numpy as np
import pytest
import torch

import clef_synth as S
from clef_synth.configs import Config, Projection
from gpu_util import bf16_dev, bf16_host
from w8a8_quantized_projections_gb300.layer import QuantizedLayer

pytestmark = pytest.mark.gpu


def small_layer(scheme, lora_rank):
    proj = [Projection("q", 1024, 1024, act="x_attn"), Projection("k", 1024, 256, act="x_attn"),
            Projection("v", 1024, 256, act="x_attn"), Projection("o", 1024, 1024, act="x_o"),
            Projection("gateup", 1024, 1536, kind="gateup", act="x_mlp"),
            Projection("down", 1536, 1024, act="x_down", chained=True)]
    return Config(90, f"graph-{scheme}", 300, scheme, proj, lora_rank=lora_rank)


def snapshot(out):
    return {k: bf16_host(v) for k, v in out.items()}


@pytest.mark.parametrize("scheme,lora_rank", [("int8", None), ("int8", 64), ("fp8", None)])
def test_graph_replay_matches_eager(scheme, lora_rank):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    cfg = small_layer(scheme, lora_rank)
    acts_np, weights_np, lora_np = S.layer_inputs(cfg, seed=3)
    weights = {k: (bf16_dev(W), bf16_dev(b)) for k, (W, b) in weights_np.items()}
    lora = {k: (bf16_dev(A), bf16_dev(B)) for k, (A, B) in lora_np.items()}
    acts = {k: bf16_dev(x) for k, x in acts_np.items()}
    layer = QuantizedLayer(cfg, weights, lora or None)
    eager = snapshot(layer.step(acts))
    torch.cuda.synchronize()

    layer.capture(acts)
    for v in layer.out.values():
        v.zero_()
    replayed = snapshot(layer.replay())
    torch.cuda.synchronize()
    assert eager.keys() == replayed.keys()
    for k in eager:
        assert np.array_equal(eager[k], replayed[k]), k

    # new inputs, refilled in place: the replay follows them
    for name, x in acts.items():
        x.copy_(bf16_dev(S.activation(4, f"graph/{name}", x.shape[0], x.shape[1])))
    replay2 = snapshot(layer.replay())
    eager2 = snapshot(layer.step(acts))
    torch.cuda.synchronize()
    for k in eager2:
        assert np.array_equal(eager2[k], replay2[k]), k
        assert not np.array_equal(eager2[k], eager[k]), k
