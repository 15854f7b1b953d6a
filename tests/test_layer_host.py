"""Host logic of the layer runner (no GPU): which projections are packed into one
GEMM launch, and the step's work accounting used by the benchmark."""
import pytest

import clef_synth as S

layer = pytest.importorskip("w8a8_quantized_projections_gb300.layer")


def _weights(cfg, bias=True):
    return {p.name: (object(), object() if bias else None) for p in cfg.projections}


def test_q_k_v_pack_into_one_launch():
    cfg = S.workload("int8-layer-27b-m2270")
    groups = layer._groups(cfg.projections, _weights(cfg))
    names = [[p.name for p in g] for g in groups]
    assert names == [["q", "k", "v"], ["o"], ["gateup"], ["down"]]
    assert layer._unit_name(groups[0]) == "q+k+v"


def test_packing_needs_the_same_input_and_bias_presence():
    cfg = S.workload("int8-layer-27b-m2270")
    w = _weights(cfg)
    w["k"] = (object(), None)     # k without bias: packed with neither q nor v
    names = [[p.name for p in g] for g in layer._groups(cfg.projections, w)]
    assert names[:4] == [["q"], ["k"], ["v"], ["o"]]
    w = _weights(cfg, bias=False)  # none with bias: q, k, v pack again
    names = [[p.name for p in g] for g in layer._groups(cfg.projections, w)]
    assert names[0] == ["q", "k", "v"]


def test_gateup_and_chained_down_are_never_packed():
    for cfg in S.CONFIGS.values():
        for g in layer._groups(cfg.projections, _weights(cfg)):
            if len(g) > 1:
                assert all(p.kind == "linear" and not p.chained for p in g)
                assert len({(p.act, p.K) for p in g}) == 1


def test_gemm_ops_count_each_projection_once():
    cfg = S.workload("int8-mlp-27b-m1502")
    # gate/up: 2 * M * (2 * 17408) * 5120; down: 2 * M * 5120 * 17408
    assert cfg.gemm_ops() == 2 * 1502 * 2 * 17408 * 5120 + 2 * 1502 * 5120 * 17408


def test_workloads_resolve_by_name_and_position():
    for i, cfg in S.CONFIGS.items():
        assert S.workload(cfg.name) is cfg
        assert S.workload(i) is cfg and S.workload(str(i)) is cfg
    with pytest.raises(KeyError):
        S.workload("no-such-workload")
