"""Full-size parity of the five workloads, in the launch configuration the
benchmark times (the same QuantizedLayer step).  The GPU runs every row; the
oracle checks sampled rows one by one (and the complete quantizer outputs
where that is cheap), each stage fed the GPU's own previous-stage output so
that errors do not compound: codes, scales and INT8 outputs bit-exact /
1 ulp, FP8 outputs within 1e-2 RMS + 1 ulp, LoRA within the derived
accumulation bound."""
import numpy as np
import pytest
import torch

import clef_synth as S
import w8a8_quantized_projections_gb300 as clef
from gpu_util import THREADS, assert_bf16_within, bf16_dev, bf16_host, bf16_ulp, host, par_rows
from w8a8_quantized_projections_gb300.layer import QuantizedLayer

pytestmark = pytest.mark.gpu

# rows checked per 128-row block (one CTA's tile rows, TMEM lanes 0..127): the
# first and last (so both rows at every 256-row CTA-pair boundary) and one in
# each middle lane quadrant; every row block is covered, so every stream-K
# split tile and the partial last block are checked in the layer's own launches
BLOCK_OFFSETS = (0, 37, 86, 127)


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    yield
    assert clef.poll_status() == 0


def sample(M):
    """Rows 128 b + o for every block b and offset o (clipped to the last row),
    whole rows so that every column tile is covered."""
    rows = [min(M - 1, 128 * b + o) for b in range(-(-M // 128)) for o in BLOCK_OFFSETS]
    return np.unique(np.array(rows, dtype=np.int64))


def prow(fn, *arrays):
    """fn over the sampled rows in threads: every array argument is row-sliced."""
    return par_rows(lambda a, b: fn(*[x[a:b] for x in arrays]), arrays[0].shape[0])


def lora_y_bound(t_ref, B, y_ref, K, r_pad, x, A):
    """Bound on |y_gpu - y_oracle| when neither side's t is shared: the final
    rounding (1 ulp), t's own error (1 ulp + 2 gamma_K sum|xA|) carried through
    |B|, and stage 2's fp32 accumulation (2 gamma_r sum|tB|)."""
    gk = (K / 16 + 2) * 2.0 ** -23
    gr = (r_pad / 16 + 2) * 2.0 ** -23
    tv = S.bf16_bits_to_f64(t_ref)[:, :A.shape[0]]
    xa = np.abs(S.bf16_bits_to_f64(x)) @ np.abs(S.bf16_bits_to_f64(A)).T
    terr = bf16_ulp(tv) + 2 * gk * xa
    Bv = np.abs(S.bf16_bits_to_f64(B))
    return (2 * bf16_ulp(S.bf16_bits_to_f64(y_ref)) + terr @ Bv.T + 2 * gr * (np.abs(tv) @ Bv.T))


@pytest.mark.parametrize("name,pack", [("int8-linear-m298-2048x2048", True),
                                       ("int8-mlp-27b-m1502", True),
                                       ("int8-layer-27b-m2270", True),
                                       ("fp8-layer-9b-m1502", True),
                                       ("int8-layer-27b-m24032-lora256", True),
                                       ("fp8-layer-9b-m1502", False)])
def test_workload_full_size(orc, name, pack):
    cfg = S.workload(name)
    fp8 = cfg.scheme == "fp8"
    acts_np, weights_np, lora_np = S.layer_inputs(cfg, seed=0)
    weights = {k: (bf16_dev(W), bf16_dev(b)) for k, (W, b) in weights_np.items()}
    lora = {k: (bf16_dev(A), bf16_dev(B)) for k, (A, B) in lora_np.items()}
    acts = {k: bf16_dev(x) for k, x in acts_np.items()}
    layer = QuantizedLayer(cfg, weights, lora or None, pack_shared_input=pack)
    if pack and {"q", "k", "v"} <= {p.name for p in cfg.projections}:
        assert [len(g) for g in layer.groups][0] == 3, "q, k and v packed into one GEMM"
    out = layer.step(acts)
    torch.cuda.synchronize()
    rows = sample(cfg.M)

    qfn = (lambda x: orc.quant_fp8(x)) if fp8 else orc.quant_int8_h128
    # weights: the GPU's weight codes equal the oracle's (bit-exact), oracle's used below
    qw = {}
    for name, (W, _) in weights_np.items():
        qw[name] = par_rows(lambda a, b: qfn(W[a:b]), W.shape[0])
        gq, gs = layer.w[name][0], layer.w[name][1]
        assert np.array_equal(host(gs), qw[name][1]), f"{name} weight scales"
        assert np.array_equal(host(gq).view(qw[name][0].dtype), qw[name][0]), f"{name} weight codes"

    # activation codes: complete comparison when small, sampled rows otherwise
    for name, x in acts_np.items():
        gq, gs = layer.q[name]
        sel = slice(None) if cfg.M * x.shape[1] <= 64 << 20 else rows
        rq, rs = par_rows(lambda a, b: qfn(x[sel][a:b]), x[sel].shape[0])
        assert np.array_equal(host(gs)[sel], rs), f"{name} scales"
        assert np.array_equal(host(gq)[sel].view(rq.dtype), rq), f"{name} codes"

    h_gpu = None
    for p in cfg.projections:
        wq, ws = qw[p.name]
        bias = weights_np[p.name][1]
        if p.chained:
            # quantizer fed the GPU's own h; then the projection fed those codes
            h_rows = bf16_host(h_gpu)[rows]
            rq, rs = prow(qfn, h_rows)
            gq, gs = layer.q[p.act]
            assert np.array_equal(host(gs)[rows], rs), "chained scales"
            assert np.array_equal(host(gq)[rows].view(rq.dtype), rq), "chained codes"
        else:
            gq, gs = layer.q[p.act]
            rq = host(gq)[rows]
            rs = host(gs)[rows]
        if p.kind == "gateup" and lora:
            # the packed base gate|up values (bit-exact INT8 linear; the unfused
            # path keeps them in a buffer, the fused one never writes them)
            lin = orc.fp8_linear if fp8 else orc.int8_linear
            base = prow(lambda q_, s_: lin(q_, s_, wq, ws, bias), rq, rs)
            if p.name + "/packed" in out:
                packed = bf16_host(out[p.name + "/packed"])[rows]
                assert np.array_equal(packed, base), "packed gate/up base"
            packed = base
            # the adapters' adds, through lora_add on the sampled rows (row-invariant
            # kernels), against the oracle; then the unfused SwiGLU against the oracle
            x = acts_np[p.act][rows]
            upd = bf16_dev(packed)
            for half, sl in (("gate", slice(0, p.N)), ("up", slice(p.N, 2 * p.N))):
                A, B = lora_np[p.name + "/" + half]
                clef.lora_add(bf16_dev(x), bf16_dev(A), bf16_dev(B), upd[:, sl])
                t_ref = prow(lambda x_: orc.lora_t(x_, A), x)
                y_ref = prow(lambda t_, b_: orc.lora_y(t_, B, b_), t_ref, np.ascontiguousarray(base[:, sl]))
                tol = lora_y_bound(t_ref, B, y_ref, p.K, clef.lora_pad(A.shape[0]), x, A)
                d = np.abs(S.bf16_bits_to_f64(bf16_host(upd)[:, sl]) - S.bf16_bits_to_f64(y_ref))
                assert np.all(d <= tol), f"{p.name}/{half} lora: excess {(d - tol).max():.3g}"
            h_unfused = bf16_host(clef.swiglu_bf16(upd))
            assert_bf16_within(h_unfused, orc.swiglu_bf16(bf16_host(upd)), 1.0, "unfused swiglu")
            # the fused LoRA gate/up + SwiGLU of the step gives the same values
            h = bf16_host(out[p.name])[rows]
            assert np.array_equal(S.bf16_bits_to_f64(h), S.bf16_bits_to_f64(h_unfused)), "fused lora swiglu"
            h_gpu = out[p.name]
        elif p.kind == "gateup":
            h = bf16_host(out[p.name])[rows]
            gfn = orc.fp8_gateup_swiglu if fp8 else orc.int8_gateup_swiglu
            ref = prow(lambda q_, s_: gfn(q_, s_, wq, ws, bias), rq, rs)
            if fp8:
                from test_gpu_parity import assert_rms_close
                assert_rms_close(h, ref, 1e-2, p.name)
            else:
                assert_bf16_within(h, ref, 1.0, p.name)
            h_gpu = out[p.name]
        else:
            y = bf16_host(out[p.name])[rows]
            lin = orc.fp8_linear if fp8 else orc.int8_linear
            ref = prow(lambda q_, s_: lin(q_, s_, wq, ws, bias), rq, rs)
            if lora and p.name in lora_np:
                A, B = lora_np[p.name]
                x = acts_np[p.act][rows]
                t_ref = prow(lambda x_: orc.lora_t(x_, A), x)
                y_ref = prow(lambda t_, r_: orc.lora_y(t_, B, r_), t_ref, ref)
                tol = lora_y_bound(t_ref, B, y_ref, p.K, clef.lora_pad(A.shape[0]), x, A)
                d = np.abs(S.bf16_bits_to_f64(y) - S.bf16_bits_to_f64(y_ref))
                assert np.all(d <= tol), f"{p.name} lora: excess {(d - tol).max():.3g}"
            elif fp8:
                from test_gpu_parity import assert_rms_close
                assert_rms_close(y, ref, 1e-2, p.name)
            else:
                assert np.array_equal(y, ref), f"{p.name}: INT8 linear not bit-exact"
    del layer, acts, weights
    torch.cuda.empty_cache()
