"""INT8 stream-K: with a workspace bound to the stream, GEMMs whose last wave
of whole tiles would leave CTA pairs idle keep their whole waves and deal the
remaining tiles' k-blocks to the pairs in even runs; the pieces of a tile meet
as exact int32 partial sums.  Every output must equal the unsplit launch's
bytes (and the oracle's)."""
import numpy as np
import pytest
import torch

import w8a8_quantized_projections_gb300 as clef
from gpu_util import dev, host, par_rows

pytestmark = pytest.mark.gpu

COUNTER_BYTES = 4096 * 2 * 8 * 4


@pytest.fixture(autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")


def codes(seed, rows, K):
    rng = np.random.default_rng(seed)
    return rng.integers(-127, 128, (rows, K)).astype(np.int8)


def bound_workspace(stream=None):
    ws = torch.zeros(clef.gemm_workspace_bytes(), dtype=torch.uint8, device="cuda")
    clef.bind_workspace(ws, stream)
    return ws


# (M, N, K) on 76 CTA pairs: 120 tiles (one whole wave, 44 tiles split); K
# of 273 k-blocks (runs end off the 16-k-block chunk grid); 88 tiles with 12
# split into two 16-k-block runs each; 180 tiles (two whole waves, 28 split);
# 120 tiles whose last column tile is partial (N = 5000); 8 and 4 tiles (under
# an eighth of a wave: every tile split in runs of 8 or more k-blocks); 48 tiles
# (under one wave: not split); 76 tiles (a full wave: not split)
SHAPES = [(1502, 5120, 17408), (1502, 5120, 17472), (1024, 5632, 2048), (2270, 5120, 6144),
          (1502, 5000, 5120), (200, 2048, 8192), (130, 1024, 4096), (300, 6144, 5120),
          (1024, 4864, 1024)]


@pytest.mark.parametrize("M,N,K", SHAPES)
def test_stream_k_s32_equals_unsplit_and_oracle(orc, M, N, K):
    qx, qw = codes(M + N, M, K), codes(K + 1, N, K)
    qx_d, qw_d = dev(qx), dev(qw)
    plain = clef.w8a8_gemm_s32(qx_d, qw_d)
    ws = bound_workspace()
    try:
        for _ in range(3):   # repeated launches reuse the zeroed counters
            split = clef.w8a8_gemm_s32(qx_d, qw_d)
            assert torch.equal(split, plain)
        torch.cuda.synchronize()
        assert int(ws[:COUNTER_BYTES].count_nonzero()) == 0, "counters must be zero between launches"
    finally:
        clef.bind_workspace(None)
    rows = np.unique(np.r_[0:3, M // 2, M - 3:M])
    ref = par_rows(lambda a, b: orc.int8_gemm_acc(qx[rows][a:b], qw), len(rows))
    assert np.array_equal(host(plain)[rows], ref)


def test_stream_k_scale_bias_equals_unsplit(orc):
    """The scale/bias epilogue on the 1,502-token down projection shape."""
    M, N, K = 1502, 5120, 17408
    qx, qw = codes(3, M, K), codes(4, N, K)
    rng = np.random.default_rng(5)
    sx = torch.tensor(rng.random(M, dtype=np.float32) * 1e-3, device="cuda")
    sw = torch.tensor(rng.random(N, dtype=np.float32) * 1e-3, device="cuda")
    b = torch.tensor(rng.standard_normal(N, dtype=np.float32), device="cuda").to(torch.bfloat16)
    qx_d, qw_d = dev(qx), dev(qw)
    plain = clef.w8a8_linear(qx_d, sx, qw_d, sw, b)
    ws = bound_workspace()
    try:
        split = clef.w8a8_linear(qx_d, sx, qw_d, sw, b)
    finally:
        clef.bind_workspace(None)
    assert torch.equal(split.view(torch.int16), plain.view(torch.int16))
    del ws


def test_stream_k_two_streams_own_workspaces():
    """Launches on two streams that overlap, each stream with its own
    workspace, give the unsplit bytes on both."""
    M, N, K = 1502, 5120, 17408
    qx_d, qw_d = dev(codes(6, M, K)), dev(codes(7, N, K))
    plain = clef.w8a8_gemm_s32(qx_d, qw_d)
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    ws1, ws2 = bound_workspace(s1), bound_workspace(s2)
    try:
        outs = []
        torch.cuda.synchronize()
        for s in (s1, s2, s1, s2):
            with torch.cuda.stream(s):
                outs.append(clef.w8a8_gemm_s32(qx_d, qw_d))
        torch.cuda.synchronize()
        for o in outs:
            assert torch.equal(o, plain)
    finally:
        clef.bind_workspace(None, s1)
        clef.bind_workspace(None, s2)
    del ws1, ws2


def test_unbound_stream_never_splits_and_unbind_works():
    """A workspace bound to another stream is not used; after unbinding,
    launches run unsplit (their counters stay untouched)."""
    M, N, K = 300, 6144, 5120
    qx_d, qw_d = dev(codes(8, M, K)), dev(codes(9, N, K))
    other = torch.cuda.Stream()
    ws = bound_workspace(other)
    ws[:COUNTER_BYTES].fill_(0)
    ref = clef.w8a8_gemm_s32(qx_d, qw_d)
    clef.bind_workspace(None, other)
    torch.cuda.synchronize()
    assert int(ws.count_nonzero()) == 0, "a workspace bound to another stream was written"
    assert torch.equal(clef.w8a8_gemm_s32(qx_d, qw_d), ref)


@pytest.mark.parametrize("M,N,K", [(1024, 2560, 4096), (300, 2048, 4096)])
def test_stream_k_swiglu_equals_unsplit(M, N, K):
    """The fused gate/up SwiGLU launches never split (their kernel has no
    split path); a bound workspace leaves their bytes and the counters as
    they were: 80 tiles of 256 rows x 128 h columns and 32 tiles."""
    rng = np.random.default_rng(M)
    qx_d = dev(codes(10, M, K))
    qw_d = dev(codes(11, 2 * N, K))
    sx = torch.tensor(rng.random(M, dtype=np.float32) * 1e-3, device="cuda")
    sw = torch.tensor(rng.random(2 * N, dtype=np.float32) * 1e-3, device="cuda")
    b = torch.tensor(rng.standard_normal(2 * N, dtype=np.float32), device="cuda").to(torch.bfloat16)
    plain = clef.w8a8_gateup_swiglu(qx_d, sx, qw_d, sw, b)
    ws = bound_workspace()
    try:
        split = clef.w8a8_gateup_swiglu(qx_d, sx, qw_d, sw, b)
        torch.cuda.synchronize()
        assert int(ws[:COUNTER_BYTES].count_nonzero()) == 0
    finally:
        clef.bind_workspace(None)
    assert torch.equal(split.view(torch.int16), plain.view(torch.int16))


# Banded tile order (row blocks ordered in bands whose activations fit 24 MB
# of L2, every column block of a band before the next band): K = 17408 gives
# bands of at most 5 row blocks; M = 2800 has 11 row blocks (bands 4, 4, 3),
# M = 6000 24 (5, 5, 5, 5, 4) and 24,032 rows 94 (bands of 5, the last of 4;
# the full-size workload tests).  With N =
# 2048 the 2,800-row launch has 88 tiles for 76 pairs (stream-K splits the
# last 12); every row block's first and last row and both rows at each CTA
# pair boundary are compared with the oracle's exact int32 sums.
@pytest.mark.parametrize("M,N,K,split", [(2800, 2048, 17408, False), (2800, 2048, 17408, True),
                                         (6000, 512, 17408, False)])
def test_banded_order_s32_equals_oracle(orc, M, N, K, split):
    qx, qw = codes(M + 7, M, K), codes(K + 7, N, K)
    qx_d, qw_d = dev(qx), dev(qw)
    ws = bound_workspace() if split else None
    try:
        got = host(clef.w8a8_gemm_s32(qx_d, qw_d))
    finally:
        if split:
            clef.bind_workspace(None)
    rows = np.unique(np.r_[np.arange(0, M, 128), np.minimum(np.arange(127, M + 127, 128), M - 1),
                           np.arange(255, M, 256), np.arange(256, M, 256)])
    ref = par_rows(lambda a, b: orc.int8_gemm_acc(qx[rows][a:b], qw), len(rows))
    assert np.array_equal(got[rows], ref)


# FP8 linear with K >= 8192: every tile sums its K as two fixed halves; with a
# workspace bound, a last wave that fits twice in the pairs runs as halves on
# two pairs (1502 x 4096 x 12288: 96 tiles for 76 pairs, 20 halved; 257 x
# 4096 x 8192: 32 tiles under one wave, all halved).  The bytes equal the
# unsplit launch's, and a call's rows equal the same rows called alone (100
# rows: single CTAs, the same halves), and sampled rows meet the oracle's FP8
# bar.
@pytest.mark.parametrize("M,N,K", [(1502, 4096, 12288), (257, 4096, 8192)])
def test_fp8_halves_split_equals_unsplit_and_rows(orc, M, N, K):
    import clef_synth as S
    from gpu_util import bf16_dev, bf16_host
    from test_gpu_parity import assert_rms_close
    x = S.activation(0, f"t/f8h/{M}x{N}x{K}/x", M, K)
    w = S.weight(0, f"t/f8h/{M}x{N}x{K}/w", N, K)
    b = S.bias(0, f"t/f8h/{M}x{N}x{K}/b", N)
    qx, sx = clef.quant_act(bf16_dev(x), "fp8")
    qw, sw = clef.quant_act(bf16_dev(w), "fp8")
    bd = bf16_dev(b)
    plain = clef.fp8_linear(qx, sx, qw, sw, bd)
    ws = bound_workspace()
    try:
        for _ in range(3):
            split = clef.fp8_linear(qx, sx, qw, sw, bd)
            assert torch.equal(split.view(torch.int16), plain.view(torch.int16))
        torch.cuda.synchronize()
        assert int(ws[:COUNTER_BYTES].count_nonzero()) == 0
    finally:
        clef.bind_workspace(None)
    full = host(plain.view(torch.int16))
    for a in (0, M // 2, M - 100):
        part = clef.fp8_linear(qx[a:a + 100].contiguous(), sx[a:a + 100].contiguous(), qw, sw, bd)
        assert np.array_equal(host(part.view(torch.int16)), full[a:a + 100]), a
    rows = np.unique(np.r_[0:2, M // 2, M - 2:M])
    qxr, sxr = orc.quant_fp8(x[rows])
    qwh, swh = par_rows(lambda a, c: orc.quant_fp8(w[a:c]), N)
    ref = orc.fp8_linear(qxr, sxr, qwh, swh, b)
    assert_rms_close(full[rows].view(np.uint16), ref, 1e-2, "fp8_linear halves")


# LoRA x A^T with K >= 6144: every tile sums its K as four fixed parts, in
# CTA-pair and single-CTA tiles alike; with a workspace bound, a last wave that
# fits four times in the pairs runs as parts on four pairs each (1,502 x 17408
# -> 256: 6 tiles under one wave, split into 24 parts; 19,712 x 6144 -> 256:
# 77 tiles, one whole wave and one tile in parts; 300 x 8192 -> 64: 64-wide
# single-CTA tiles).  The bytes equal the unsplit launch's, a call's rows equal
# the same rows called alone (100 rows: single CTAs), and sampled rows meet the
# oracle within the fp32 accumulation bound.
@pytest.mark.parametrize("M,K,r", [(1502, 17408, 256), (19712, 6144, 256), (300, 8192, 64)])
def test_lora_shrink_parts_split_equals_unsplit_and_rows(orc, M, K, r):
    import clef_synth as S
    from gpu_util import bf16_dev, bf16_ulp
    from test_gpu_parity import lora_bound
    x = S.activation(0, f"t/lsp/{M}x{K}/x", M, K)
    A, _ = S.lora_pair(0, f"t/lsp/{M}x{K}", r, K, 8)
    xd, Ad = bf16_dev(x), bf16_dev(A)
    plain = clef.lora_shrink(xd, Ad)
    ws = bound_workspace()
    try:
        for _ in range(3):
            split = clef.lora_shrink(xd, Ad)
            assert torch.equal(split.view(torch.int16), plain.view(torch.int16))
        torch.cuda.synchronize()
        assert int(ws[:COUNTER_BYTES].count_nonzero()) == 0
    finally:
        clef.bind_workspace(None)
    full = host(plain.view(torch.int16))
    for a in (0, M // 2, M - 100):
        part = clef.lora_shrink(xd[a:a + 100].contiguous(), Ad)
        assert np.array_equal(host(part.view(torch.int16)), full[a:a + 100]), a
    rows = np.unique(np.r_[0:2, M // 2, M - 2:M])
    t_ref = orc.lora_t(x[rows], A)
    t = full[rows].view(np.uint16)[:, :r]
    tol = bf16_ulp(S.bf16_bits_to_f64(t_ref[:, :r])) + 2 * lora_bound(x[rows], A, K)
    d = np.abs(S.bf16_bits_to_f64(t) - S.bf16_bits_to_f64(t_ref[:, :r]))
    assert np.all(d <= tol), f"t: worst excess {(d - tol).max():.3g}"
    assert np.all(full[:, r:clef.lora_pad(r)] == 0), "padding columns of t must be exact zeros"
