"""The runtime LoRA expand fused into the INT8 GEMMs (the pull request's
y = bf16(y + bf16(x A^T) B^T) with y the rounded base projection).

The fused calls must give the bytes of the unfused chains they replace --
clef_w8a8_linear then clef_lora_expand_add, or the packed clef_w8a8_linear
then clef_lora_gateup_swiglu -- on CTA-pair tiles (M > 128) and single
tiles, ragged M and N, ranks that need padding, several tiles per CTA pair,
packed projections with several adapters (column segments), and rows checked
against the oracle through the same chain.  A layer with the fused path
equals one without it, and the fused calls keep a row's bits independent of
the call's row count."""
import numpy as np
import pytest
import torch

import clef_synth as S
import w8a8_quantized_projections_gb300 as clef
from gpu_util import bf16_dev, bf16_host

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    yield
    assert clef.poll_status() == 0


def _eq(a, b, what):
    assert torch.equal(a.view(torch.int16), b.view(torch.int16)), \
        f"{what}: {int((a.view(torch.int16) != b.view(torch.int16)).sum())} of {a.numel()} differ"


def _codes(tag, M, N, K, bias=True):
    x = bf16_dev(S.activation(0, f"t/fl/{tag}/x", M, K))
    w = bf16_dev(S.weight(0, f"t/fl/{tag}/w", N, K))
    b = bf16_dev(S.bias(0, f"t/fl/{tag}/b", N)) if bias else None
    qx, sx = clef.quant_act(x, "int8_h128")
    qw, sw = clef.quant_act(w, "int8_h128")
    return x, qx, sx, qw, sw, b


@pytest.mark.parametrize("M,N,K,r,bias", [(300, 1024, 2048, 256, True), (130, 264, 1024, 48, False),
                                          (1, 8, 128, 8, True), (600, 2560, 5120, 256, True),
                                          (257, 512, 17408, 64, True),
                                          (2048, 8192, 1024, 256, True)])   # 256 tiles: several per pair
def test_linear_lora_equals_linear_then_expand(M, N, K, r, bias):
    x, qx, sx, qw, sw, b = _codes(f"lin{M}", M, N, K, bias)
    A, B = (bf16_dev(v) for v in S.lora_pair(0, f"t/fl/lin{M}/l", r, K, N))
    t = clef.lora_shrink(x, A)
    ref = clef.w8a8_linear(qx, sx, qw, sw, b)
    clef.lora_expand_add(t, B, ref)
    got = clef.w8a8_linear_lora(qx, sx, qw, sw, b, t, B)
    _eq(got, ref, "fused linear")


@pytest.mark.parametrize("M", [300, 100])
def test_linear_lora_segments(M):
    """A packed q|k|v-shaped unit: three adapters' B factors stacked in
    output order, t of the three adapters side by side, a middle projection
    without an adapter (zero B rows)."""
    Nq, Nk, Nv, K, r = 768, 256, 512, 1024, 64
    N = Nq + Nk + Nv
    x, qx, sx, qw, sw, b = _codes(f"seg{M}", M, N, K)
    Aq, Bq = (bf16_dev(v) for v in S.lora_pair(0, f"t/fl/seg{M}/q", r, K, Nq))
    Av, Bv = (bf16_dev(v) for v in S.lora_pair(0, f"t/fl/seg{M}/v", r, K, Nv))
    t = clef.lora_shrink(x, torch.cat([Aq, Av]))         # [M][128]: t_q | t_v
    B = torch.zeros((N, r), dtype=torch.bfloat16, device="cuda")
    B[:Nq] = Bq
    B[Nq + Nk:] = Bv
    got = clef.w8a8_linear_lora(qx, sx, qw, sw, b, t, B, segments=[(Nq, 0), (Nq + Nk, 0), (N, 64)])
    ref = clef.w8a8_linear(qx, sx, qw, sw, b)
    clef.lora_expand_add(t[:, :64], Bq, ref[:, :Nq])
    clef.lora_expand_add(t[:, 64:], Bv, ref[:, Nq + Nk:])
    _eq(got, ref, "segments")


@pytest.mark.parametrize("M,N,K,r", [(300, 512, 1024, 256), (130, 264, 2048, 48), (1, 8, 128, 8),
                                     (600, 1280, 5120, 256), (2048, 4096, 1024, 256)])
def test_gateup_swiglu_lora_equals_unfused(M, N, K, r):
    x, qx, sx, qw, sw, b = _codes(f"gu{M}", M, 2 * N, K)
    Ag, Bg = (bf16_dev(v) for v in S.lora_pair(0, f"t/fl/gu{M}/g", r, K, N))
    Au, Bu = (bf16_dev(v) for v in S.lora_pair(0, f"t/fl/gu{M}/u", r, K, N))
    rp = clef.lora_pad(r)
    A = torch.zeros((2 * rp, K), dtype=torch.bfloat16, device="cuda")
    A[:r], A[rp:rp + r] = Ag, Au
    t = clef.lora_shrink(x, A)
    ygu = clef.w8a8_linear(qx, sx, qw, sw, b)
    ref = clef.lora_gateup_swiglu(x, Ag, Bg, Au, Bu, ygu)
    got = clef.w8a8_gateup_swiglu_lora(qx, sx, qw, sw, b, t, Bg, Bu)
    _eq(got, ref, "fused gate/up")


def test_fused_rows_match_oracle(orc):
    """Sampled rows of a fused linear against the oracle's chain (INT8 linear,
    LoRA t, LoRA y), within the derived LoRA bound."""
    from test_gpu_configs import lora_y_bound
    M, N, K, r = 300, 512, 2048, 256
    x, qx, sx, qw, sw, b = _codes("orc", M, N, K)
    xn = S.activation(0, "t/fl/orc/x", M, K)
    An, Bn = S.lora_pair(0, "t/fl/orc/l", r, K, N)
    t = clef.lora_shrink(x, bf16_dev(An))
    y = bf16_host(clef.w8a8_linear_lora(qx, sx, qw, sw, b, t, bf16_dev(Bn)))
    rows = np.array([0, 1, 127, 128, 255, 256, 299])
    base = orc.int8_linear(qx.cpu().numpy()[rows], sx.cpu().numpy()[rows], qw.cpu().numpy(),
                           sw.cpu().numpy(), S.bias(0, "t/fl/orc/b", N))
    t_ref = orc.lora_t(xn[rows], An)
    y_ref = orc.lora_y(t_ref, Bn, base)
    tol = lora_y_bound(t_ref, Bn, y_ref, K, clef.lora_pad(r), xn[rows], An)
    d = np.abs(S.bf16_bits_to_f64(y[rows]) - S.bf16_bits_to_f64(y_ref))
    assert np.all(d <= tol), f"excess {(d - tol).max():.3g}"


def test_fused_row_invariance():
    """600 rows at once equal pieces of 1..255 rows."""
    from test_gpu_parity import pieces
    M, N, K, r = 600, 1024, 1024, 64
    x, qx, sx, qw, sw, b = _codes("inv", M, N, K)
    A1, B1 = (bf16_dev(v) for v in S.lora_pair(0, "t/fl/inv/1", r, K, N // 2))
    A2, B2 = (bf16_dev(v) for v in S.lora_pair(0, "t/fl/inv/2", r, K, N // 2))
    t = clef.lora_shrink(x, torch.cat([A1, A2]))
    B = torch.cat([B1, B2])
    segs = [(N // 2, 0), (N, 64)]
    whole = clef.w8a8_linear_lora(qx, sx, qw, sw, b, t, B, segments=segs)
    part = torch.empty_like(whole)
    for a, c in pieces(M):
        clef.w8a8_linear_lora(qx[a:c], sx[a:c], qw, sw, b, t[a:c], B, y=part[a:c], segments=segs)
    _eq(whole, part, "linear")
    Ag, Bg = (bf16_dev(v) for v in S.lora_pair(0, "t/fl/inv/g", r, K, N // 2))
    Au, Bu = (bf16_dev(v) for v in S.lora_pair(0, "t/fl/inv/u", r, K, N // 2))
    t = clef.lora_shrink(x, torch.cat([Ag, Au]))
    whole = clef.w8a8_gateup_swiglu_lora(qx, sx, qw, sw, b, t, Bg, Bu)
    part = torch.empty_like(whole)
    for a, c in pieces(M):
        clef.w8a8_gateup_swiglu_lora(qx[a:c], sx[a:c], qw, sw, b, t[a:c], Bg, Bu, h=part[a:c])
    _eq(whole, part, "gate/up")


def test_layer_fused_equals_unfused():
    """A 27B-shaped layer (q|k|v packed, o, gate/up, down) at 300 tokens with
    rank-256 adapters on every projection: the fused step's outputs equal
    the unfused step's byte for byte."""
    from clef_synth.configs import Config, Projection
    from w8a8_quantized_projections_gb300.layer import QuantizedLayer
    cfg = Config(91, "fused-test-27b-m300", 300, "int8", [
        Projection("q", 1024, 1536, act="x_attn"), Projection("k", 1024, 256, act="x_attn"),
        Projection("v", 1024, 256, act="x_attn"), Projection("o", 1536, 1024, act="x_o"),
        Projection("gateup", 1024, 2816, kind="gateup", act="x_mlp"),
        Projection("down", 2816, 1024, act="h", chained=True)], lora_rank=256)
    acts_np, weights_np, lora_np = S.layer_inputs(cfg, seed=0)
    weights = {k: (bf16_dev(W), bf16_dev(b)) for k, (W, b) in weights_np.items()}
    lora = {k: (bf16_dev(A), bf16_dev(B)) for k, (A, B) in lora_np.items()}
    acts = {k: bf16_dev(x) for k, x in acts_np.items()}
    fused = QuantizedLayer(cfg, weights, lora, fuse_lora=True)
    plain = QuantizedLayer(cfg, weights, lora, fuse_lora=False)
    assert len(fused.fused) == 4, "q|k|v, o, gate/up and down fused"
    of = {k: v.clone() for k, v in fused.step(acts).items()}
    op = plain.step(acts)
    for p in cfg.projections:
        _eq(of[p.name], op[p.name], p.name)
    assert fused.poll_status() == 0
