"""GPU parity: every CUDA entry point against the CPU oracle on the same
seeded inputs, through the C ABI (via the thin Python binding).

Bars: INT8 and e4m3 codes, scales and int32 accumulators bit-exact; INT8
path bf16 outputs within 1 bf16 ulp (the scale/bias epilogue is asserted
bit-exact: it runs the same rounded operations in the same order); FP8
outputs within 1e-2 x RMS(reference) given identical codes; LoRA within the
bound derived from fp32 accumulation (see test_lora_add)."""
import numpy as np
import pytest
import torch

import clef_synth as S
import w8a8_quantized_projections_gb300 as clef
from gpu_util import (assert_bf16_within, bf16_dev, bf16_host, bf16_ulp, dev, host, par_rows,
                      ulp_diff)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    clef.library()
    yield
    assert clef.poll_status() == 0


def special_rows(x: np.ndarray) -> np.ndarray:
    """Row 0 all zero, row 1 one-hot, row 2 a single huge outlier."""
    x = x.copy()
    if x.shape[0] >= 3:
        x[0] = 0
        x[1] = 0
        x[1, 5] = S.f64_to_bf16_bits(np.array([-3.25]))[0]
        x[2, x.shape[1] // 2] = S.f64_to_bf16_bits(np.array([1.0e4]))[0]
    return x


# ------------------------------------------------------------------ quantizer

@pytest.fixture(params=[2, 0], ids=["staged", "per_row"])
def staging(request):
    """Run a quantizer test with the TMA-staged persistent kernel (wherever the
    row length allows it, whatever the row count) and with the
    one-CTA-per-row kernel."""
    clef.set_quant_staging(request.param)
    yield request.param
    clef.set_quant_staging(1)


@pytest.mark.parametrize("M,K", [(298, 2048), (1, 128), (5, 384), (130, 5120), (1502, 17408),
                                 (2270, 6144), (3, 40960), (12000, 5120), (2, 128 * 131), (4, 65536),
                                 (700, 8192), (33, 12288), (5, 128 * 71)])
def test_quant_int8_h128_bitexact(orc, staging, M, K):
    x = special_rows(S.activation(0, f"t/q8/{M}x{K}", M, K))
    q, s = clef.quant_act(bf16_dev(x), "int8_h128")
    rq, rs = par_rows(lambda a, b: orc.quant_int8_h128(x[a:b]), M)
    assert np.array_equal(host(s), rs)
    assert np.array_equal(host(q), rq)


def test_quant_strided_rows(orc, staging):
    M, K, ld = 37, 1024, 1536
    big = S.activation(0, "t/q8/strided", M, ld)
    xt = bf16_dev(big)[:, :K]
    q, s = clef.quant_act(xt, "int8_h128")
    rq, rs = orc.quant_int8_h128(np.ascontiguousarray(big[:, :K]))
    assert np.array_equal(host(q), rq) and np.array_equal(host(s), rs)


@pytest.mark.parametrize("mode", ["fp8", "fp8_h128"])
@pytest.mark.parametrize("M,K", [(1502, 4096), (7, 12288), (33, 640), (1, 128), (9, 96)])
def test_quant_fp8_bitexact(orc, staging, mode, M, K):
    if mode == "fp8_h128" and K % 128:
        pytest.skip("the rotated mode needs whole 128-blocks")
    x = special_rows(S.activation(0, f"t/q8f/{M}x{K}", M, K))
    q, s = clef.quant_act(bf16_dev(x), mode)
    rq, rs = par_rows(lambda a, b: orc.quant_fp8(x[a:b], rotate=(mode == "fp8_h128")), M)
    assert np.array_equal(host(s), rs)
    got = host(q)
    if not np.array_equal(got, rq):
        bad = np.argwhere(got != rq)
        m, k = bad[0]
        raise AssertionError(f"{len(bad)} e4m3 codes differ, first at {m},{k}: gpu {got[m, k]:#x} "
                             f"oracle {rq[m, k]:#x}")


@pytest.mark.parametrize("mode,sc", [("int8_h128", 0.0625), ("int8_h128", 0.037), ("fp8", 2.0 ** -7),
                                     ("fp8", 0.0123), ("fp8_h128", 0.0123)])
@pytest.mark.parametrize("M,K", [(300, 2048), (1502, 5120)])
def test_quant_static_bitexact(orc, staging, mode, sc, M, K):
    """Static per-tensor scale: codes (saturating) and scales bit-exact, on
    both quantizer kernels."""
    x = S.activation(0, f"t/qs/{M}x{K}", M, K)
    q, s = clef.quant_act_static(bf16_dev(x), sc, mode)
    rq, rs = par_rows(lambda a, b: orc.quant_static(x[a:b], sc, mode), M)
    assert np.array_equal(host(s), rs)
    got = host(q)
    assert np.array_equal(got.view(rq.dtype), rq)


def test_quant_empty_rows():
    x = torch.empty((0, 256), dtype=torch.bfloat16, device="cuda")
    q, s = clef.quant_act(x, "int8_h128")
    assert q.shape == (0, 256) and s.shape == (0,)


# ------------------------------------------------------------------ INT8 GEMM

def quantized(orc, name, M, N, K, seed=0):
    x = S.activation(seed, f"{name}/x", M, K)
    w = S.weight(seed, f"{name}/w", N, K)
    b = S.bias(seed, f"{name}/b", N)
    qx, sx = par_rows(lambda a, c: orc.quant_int8_h128(x[a:c]), M)
    qw, sw = par_rows(lambda a, c: orc.quant_int8_h128(w[a:c]), N)
    return x, w, b, qx, sx, qw, sw


@pytest.mark.parametrize("M,N,K", [(298, 2048, 2048), (1, 8, 16), (130, 264, 80), (257, 512, 1088),
                                   (129, 1024, 5120)])
def test_int8_gemm_s32_bitexact(orc, M, N, K):
    rng = np.random.default_rng(M * 7 + N + K)
    qx = rng.integers(-127, 128, (M, K)).astype(np.int8)
    qw = rng.integers(-127, 128, (N, K)).astype(np.int8)
    acc = host(clef.w8a8_gemm_s32(dev(qx), dev(qw)))
    ref = par_rows(lambda a, b: orc.int8_gemm_acc(qx[a:b], qw), M)
    assert np.array_equal(acc, ref)


def test_int8_gemm_s32_max_depth(orc):
    """K = 65536, the largest depth the quantizer accepts: all codes 127 give
    127 * 127 * 65536 = 1,057,030,144 (still an int32), exact through 64
    fp32 chunks; mixed signs and a random row check the rest."""
    M, N, K = 3, 24, 65536
    rng = np.random.default_rng(17)
    qx = np.full((M, K), 127, np.int8)
    qx[1] = -127
    qx[2] = rng.integers(-127, 128, K).astype(np.int8)
    qw = np.full((N, K), 127, np.int8)
    qw[5] = rng.integers(-127, 128, K).astype(np.int8)
    acc = host(clef.w8a8_gemm_s32(dev(qx), dev(qw)))
    assert acc[0, 0] == 127 * 127 * K and acc[1, 0] == -127 * 127 * K
    assert np.array_equal(acc, orc.int8_gemm_acc(qx, qw))


def test_int8_gemm_s32_adversarial(orc):
    """Sums far beyond 2^24 (the exact range of fp32) stay exact: all codes
    +-127 over K = 17408 reach +-280,773,632."""
    M, N, K = 130, 264, 17408
    rng = np.random.default_rng(11)
    qx = np.full((M, K), 127, np.int8)
    qx[1::2] = -127
    qx[5, :] = rng.choice(np.array([-127, 127], np.int8), K)
    qw = np.full((N, K), 127, np.int8)
    qw[3] = -127
    qw[7, ::3] = -127
    qw[9, :] = rng.integers(-127, 128, K).astype(np.int8)
    acc = host(clef.w8a8_gemm_s32(dev(qx), dev(qw)))
    assert acc[0, 0] == 280773632 and acc[1, 0] == -280773632
    ref = par_rows(lambda a, b: orc.int8_gemm_acc(qx[a:b], qw), M)
    assert np.array_equal(acc, ref)


@pytest.mark.parametrize("M,N,K,with_bias", [(298, 2048, 2048, True), (300, 1024, 5120, False),
                                             (5, 8, 128, True)])
def test_w8a8_linear_bitexact(orc, M, N, K, with_bias):
    x, w, b, qx, sx, qw, sw = quantized(orc, f"t/lin/{M}x{N}x{K}", M, N, K)
    bias = b if with_bias else None
    # the GPU quantizer feeds the GPU GEMM; its codes equal the oracle's (tested above)
    gqx, gsx = clef.quant_act(bf16_dev(x), "int8_h128")
    gqw, gsw = clef.quant_act(bf16_dev(w), "int8_h128")
    assert np.array_equal(host(gqx), qx) and np.array_equal(host(gqw), qw)
    y = bf16_host(clef.w8a8_linear(gqx, gsx, gqw, gsw, bf16_dev(bias) if with_bias else None))
    ref = par_rows(lambda a, c: orc.int8_linear(qx[a:c], sx[a:c], qw, sw, bias), M)
    assert np.array_equal(y, ref), f"max {ulp_diff(y, ref).max()} ulp"


def test_w8a8_linear_zero_row_gives_bias(orc):
    M, N, K = 4, 64, 256
    x = S.activation(0, "t/zero/x", M, K)
    x[2] = 0
    w = S.weight(0, "t/zero/w", N, K)
    b = S.bias(0, "t/zero/b", N)
    qx, sx = clef.quant_act(bf16_dev(x))
    qw, sw = clef.quant_act(bf16_dev(w))
    y = bf16_host(clef.w8a8_linear(qx, sx, qw, sw, bf16_dev(b)))
    assert np.array_equal(y[2], b)


@pytest.mark.parametrize("M,N,K", [(298, 1024, 2048), (130, 136, 1024), (1, 8, 128)])
def test_w8a8_gateup_swiglu(orc, M, N, K):
    x, w, b, qx, sx, qw, sw = quantized(orc, f"t/gu/{M}x{N}x{K}", M, 2 * N, K)
    h = bf16_host(clef.w8a8_gateup_swiglu(dev(qx), dev(sx), dev(qw), dev(sw), bf16_dev(b)))
    ref = par_rows(lambda a, c: orc.int8_gateup_swiglu(qx[a:c], sx[a:c], qw, sw, b), M)
    assert_bf16_within(h, ref, 1.0, "swiglu")


def test_w8a8_gateup_swiglu_wide_gate_range(orc):
    """Gate values from about -200 to +200 (gate scales spread over four
    decades), so silu meets its saturated ends: exp(-g) overflowing to
    infinity, denominators beyond 2^126, and silu(g) = g."""
    M, N, K = 130, 256, 256
    rng = np.random.default_rng(5)
    qx = rng.integers(-127, 128, (M, K)).astype(np.int8)
    qw = rng.integers(-127, 128, (2 * N, K)).astype(np.int8)
    sx = np.ones(M, np.float32)
    sw = np.empty(2 * N, np.float32)
    sw[:N] = (10.0 ** np.linspace(-6, -2.3, N)).astype(np.float32)
    sw[N:] = np.float32(1e-4)
    b = S.bias(0, "t/gu/wide/b", 2 * N)
    h = bf16_host(clef.w8a8_gateup_swiglu(dev(qx), dev(sx), dev(qw), dev(sw), bf16_dev(b)))
    ref = orc.int8_gateup_swiglu(qx, sx, qw, sw, b)
    g = (qx.astype(np.int64) @ qw[:N].T.astype(np.int64)) * sw[:N].astype(np.float64)
    assert g.min() < -90 and g.max() > 90
    assert_bf16_within(h, ref, 1.0, "swiglu wide gate")


@pytest.mark.parametrize("M,K,N,r", [(300, 1024, 512, 256), (130, 512, 264, 48), (1, 128, 8, 8),
                                     (600, 2048, 1024, 128)])
def test_lora_gateup_swiglu_equals_unfused(M, K, N, r):
    """The fused gate/up LoRA + SwiGLU call gives the values of two lora_add
    calls on the halves followed by swiglu_bf16 (the same rounded operations;
    the other adapter's columns meet zeros, which add nothing)."""
    x = bf16_dev(S.activation(0, f"t/lgu/{M}/x", M, K))
    Ag, Bg = (bf16_dev(a) for a in S.lora_pair(0, f"t/lgu/{M}/g", r, K, N))
    Au, Bu = (bf16_dev(a) for a in S.lora_pair(0, f"t/lgu/{M}/u", r, K, N))
    y = bf16_dev(S.normal_bf16(0, f"t/lgu/{M}/y", (M, 2 * N), 2.0))
    h = bf16_host(clef.lora_gateup_swiglu(x, Ag, Bg, Au, Bu, y))
    upd = y.clone()
    clef.lora_add(x, Ag, Bg, upd[:, :N])
    clef.lora_add(x, Au, Bu, upd[:, N:])
    ref = bf16_host(clef.swiglu_bf16(upd))
    assert np.array_equal(S.bf16_bits_to_f64(h), S.bf16_bits_to_f64(ref))
    assert np.array_equal(bf16_host(y), S.normal_bf16(0, f"t/lgu/{M}/y", (M, 2 * N), 2.0)), "y_gu read only"


@pytest.mark.parametrize("std", [3.0, 40.0])
def test_swiglu_bf16(orc, std):
    """Gate values N(0, std^2): std 40 reaches the saturated ends of silu
    (exp(-g) overflowing, denominators beyond 2^126, silu(g) = g)."""
    M, N = 300, 1024
    y = S.normal_bf16(0, "t/sw/y", (M, 2 * N), std)
    h = bf16_host(clef.swiglu_bf16(bf16_dev(y)))
    ref = orc.swiglu_bf16(y)
    assert_bf16_within(h, ref, 1.0, "swiglu_bf16")


# ------------------------------------------------------------------ FP8 GEMM

def fp8_quantized(orc, name, M, N, K):
    x = S.activation(0, f"{name}/x", M, K)
    w = S.weight(0, f"{name}/w", N, K)
    b = S.bias(0, f"{name}/b", N)
    gqx, gsx = clef.quant_act(bf16_dev(x), "fp8")
    gqw, gsw = clef.quant_act(bf16_dev(w), "fp8")
    qx, sx = par_rows(lambda a, c: orc.quant_fp8(x[a:c]), M)
    qw, sw = par_rows(lambda a, c: orc.quant_fp8(w[a:c]), N)
    assert np.array_equal(host(gqx), qx) and np.array_equal(host(gqw), qw)
    return b, gqx, gsx, gqw, gsw, qx, sx, qw, sw


def assert_rms_close(got_u16, ref_u16, rel=1e-2, what=""):
    """FP8 bar: |gpu - oracle| <= rel * RMS(oracle) + 1 bf16 ulp(oracle).  The
    RMS term bounds the accumulation-order difference; the ulp term is the
    final bf16 rounding, which may fall either way once the fp32 values differ
    (at |y| >= 4 one ulp, 2^-5, already exceeds 1e-2 * RMS for RMS < 3.1)."""
    g, r = S.bf16_bits_to_f64(got_u16), S.bf16_bits_to_f64(ref_u16)
    rms = np.sqrt(np.mean(r ** 2))
    d = np.abs(g - r)
    excess = d - (rel * rms + bf16_ulp(r))
    assert np.all(excess <= 0), (f"{what}: {int((excess > 0).sum())} outside, max |diff| {d.max():.3g}, "
                                 f"RMS {rms:.3g}")
    # and the accumulation difference itself is small: nearly all within one ulp
    assert np.mean(d > bf16_ulp(r)) < 1e-3, f"{what}: {np.mean(d > bf16_ulp(r)):.2e} beyond 1 ulp"


@pytest.mark.parametrize("M,N,K", [(300, 1024, 4096), (130, 264, 256), (1, 8, 128), (129, 512, 12288)])
def test_fp8_linear(orc, M, N, K):
    b, gqx, gsx, gqw, gsw, qx, sx, qw, sw = fp8_quantized(orc, f"t/f8/{M}x{N}x{K}", M, N, K)
    y = bf16_host(clef.fp8_linear(gqx, gsx, gqw, gsw, bf16_dev(b)))
    ref = par_rows(lambda a, c: orc.fp8_linear(qx[a:c], sx[a:c], qw, sw, b), M)
    assert_rms_close(y, ref, 1e-2, "fp8_linear")


@pytest.mark.parametrize("mode", ["int8_h128", "fp8"])
def test_packed_projections_equal_separate_calls(mode):
    """q|k|v packed into one GEMM (weight rows, scales and biases stacked) give
    each projection's outputs bit for bit as separate calls do."""
    M, K = 300, 1024
    widths = [768, 256, 256]
    x = S.activation(0, "t/pack/x", M, K)
    ws = [S.weight(0, f"t/pack/w{i}", n, K) for i, n in enumerate(widths)]
    bs = [S.bias(0, f"t/pack/b{i}", n) for i, n in enumerate(widths)]
    lin = clef.w8a8_linear if mode == "int8_h128" else clef.fp8_linear
    qx, sx = clef.quant_act(bf16_dev(x), mode)
    packed_w = bf16_dev(np.concatenate(ws, axis=0))
    qw, sw = clef.quant_act(packed_w, mode)
    y_packed = host(lin(qx, sx, qw, sw, bf16_dev(np.concatenate(bs))).view(torch.int16))
    c0 = 0
    for w, b, n in zip(ws, bs, widths):
        qwi, swi = clef.quant_act(bf16_dev(w), mode)
        yi = host(lin(qx, sx, qwi, swi, bf16_dev(b)).view(torch.int16))
        assert np.array_equal(yi, y_packed[:, c0:c0 + n])
        c0 += n


def test_fp8_gateup_swiglu(orc):
    M, N, K = 300, 512, 4096
    b, gqx, gsx, gqw, gsw, qx, sx, qw, sw = fp8_quantized(orc, "t/f8gu", M, 2 * N, K)
    h = bf16_host(clef.fp8_gateup_swiglu(gqx, gsx, gqw, gsw, bf16_dev(b)))
    ref = par_rows(lambda a, c: orc.fp8_gateup_swiglu(qx[a:c], sx[a:c], qw, sw, b), M)
    assert_rms_close(h, ref, 1e-2, "fp8_gateup_swiglu")


# ------------------------------------------------------------------ LoRA

def lora_bound(x_u16, A_u16, K):
    """fp32 accumulation bound: (K/16 + 2) * 2^-23 * sum_k |x_k A_jk|."""
    xa = np.abs(S.bf16_bits_to_f64(x_u16)) @ np.abs(S.bf16_bits_to_f64(A_u16)).T
    return (K / 16 + 2) * 2.0 ** -23 * xa


@pytest.mark.parametrize("M,K,N,r", [(300, 5120, 1024, 256), (130, 2048, 264, 48), (1, 128, 8, 8),
                                     (257, 1024, 512, 128)])
def test_lora_add(orc, M, K, N, r):
    x = S.activation(0, f"t/lora/{M}/x", M, K)
    A, B = S.lora_pair(0, f"t/lora/{M}", r, K, N)
    y0 = S.normal_bf16(0, f"t/lora/{M}/y", (M, N))
    r_pad = clef.lora_pad(r)
    t_dev = torch.empty((M, r_pad), dtype=torch.bfloat16, device="cuda")
    y_dev = bf16_dev(y0)
    clef.lora_add(bf16_dev(x), bf16_dev(A), bf16_dev(B), y_dev, t_scratch=t_dev)
    t = bf16_host(t_dev)
    # stage 1: t within 1 ulp of the oracle plus the fp32 accumulation bound
    t_ref = par_rows(lambda a, c: orc.lora_t(x[a:c], A), M)
    assert np.all(t[:, r:] == 0), "padding columns of t must be exact zeros"
    tol = bf16_ulp(S.bf16_bits_to_f64(t_ref[:, :r])) + 2 * lora_bound(x, A, K)
    d = np.abs(S.bf16_bits_to_f64(t[:, :r]) - S.bf16_bits_to_f64(t_ref[:, :r]))
    assert np.all(d <= tol), f"t: worst excess {(d - tol).max():.3g}"
    # stage 2, fed the GPU's t
    y = bf16_host(y_dev)
    y_ref = par_rows(lambda a, c: orc.lora_y(t[a:c], B, y0[a:c]), M)
    tol2 = bf16_ulp(S.bf16_bits_to_f64(y_ref)) + 2 * lora_bound(t, np.pad(B, ((0, 0), (0, r_pad - r))), r_pad)
    d2 = np.abs(S.bf16_bits_to_f64(y) - S.bf16_bits_to_f64(y_ref))
    assert np.all(d2 <= tol2), f"y: worst excess {(d2 - tol2).max():.3g}"


def stacked_adapters(name, K, ranks, Ns):
    """Adapters on one input: their (A, B) pairs and the A factors stacked,
    each zero-padded to a multiple of 64 rows."""
    pairs = [S.lora_pair(0, f"{name}/{i}", r, K, N) for i, (r, N) in enumerate(zip(ranks, Ns))]
    pads = [clef.lora_pad(r) for r in ranks]
    A_cat = np.zeros((sum(pads), K), np.uint16)
    o = 0
    for (A, _), p in zip(pairs, pads):
        A_cat[o:o + A.shape[0]] = A
        o += p
    return pairs, pads, A_cat


@pytest.mark.parametrize("M,K", [(300, 1024), (1, 128), (130, 2048)])
def test_lora_shrink_expand_equal_lora_add(M, K):
    """One shrink over three adapters' stacked A factors, then one expand per
    adapter from its column block of t (pitch = the stacked width), gives
    each adapter's lora_add bytes."""
    ranks, Ns = (256, 48, 128), (512, 264, 128)
    x = bf16_dev(S.activation(0, f"t/lst/{M}/x", M, K))
    pairs, pads, A_cat = stacked_adapters(f"t/lst/{M}", K, ranks, Ns)
    t = clef.lora_shrink(x, bf16_dev(A_cat))
    o = 0
    for i, ((A, B), p) in enumerate(zip(pairs, pads)):
        y0 = S.normal_bf16(0, f"t/lst/{M}/y{i}", (M, B.shape[0]))
        y_sh, y_ref = bf16_dev(y0), bf16_dev(y0)
        clef.lora_expand_add(t[:, o:o + p], bf16_dev(B), y_sh)
        clef.lora_add(x, bf16_dev(A), bf16_dev(B), y_ref)
        assert torch.equal(y_sh.view(torch.int16), y_ref.view(torch.int16)), f"adapter {i}"
        o += p


def test_lora_shrink_tile_shape_does_not_change_t(orc):
    """24,032 rows: a rank-64 and a rank-192 factor stacked (256 columns) run as
    256-wide CTA-pair tiles, the rank-64 factor alone as 64-wide single-CTA
    tiles, and 100 of the rows alone as one 256-wide single-CTA tile; every
    element of t is the same fp32 sum of the same products in the same k
    order in each, so the bytes agree.  Checked against the oracle too."""
    M, K = 24032, 128
    pairs, pads, A_cat = stacked_adapters("t/lsw", K, (64, 192), (64, 64))
    x_h = S.activation(0, "t/lsw/x", M, K)
    x = bf16_dev(x_h)
    t_cat = clef.lora_shrink(x, bf16_dev(A_cat))
    t_one = clef.lora_shrink(x, bf16_dev(pairs[0][0]))
    assert torch.equal(t_cat[:, :64].view(torch.int16), t_one.view(torch.int16))
    t_few = clef.lora_shrink(x[5000:5100], bf16_dev(A_cat))
    assert torch.equal(t_cat[5000:5100].view(torch.int16), t_few.view(torch.int16))
    A1 = pairs[1][0]
    rows = np.r_[0:200, M - 300:M]
    t_ref = orc.lora_t(x_h[rows], A1)
    t = bf16_host(t_cat[:, 64:256])[rows]
    tol = bf16_ulp(S.bf16_bits_to_f64(t_ref)) + 2 * lora_bound(x_h[rows], A1, K)
    d = np.abs(S.bf16_bits_to_f64(t) - S.bf16_bits_to_f64(t_ref))
    assert np.all(d <= tol), f"t: worst excess {(d - tol).max():.3g}"


def test_lora_rank48_equals_zero_padded_64(orc):
    """A rank-48 pair and the same pair zero-padded to 64 give identical bytes."""
    M, K, N = 64, 1024, 256
    x = bf16_dev(S.activation(0, "t/l48/x", M, K))
    A, B = S.lora_pair(0, "t/l48", 48, K, N)
    y0 = S.normal_bf16(0, "t/l48/y", (M, N))
    y48, y64 = bf16_dev(y0), bf16_dev(y0)
    clef.lora_add(x, bf16_dev(A), bf16_dev(B), y48)
    A64 = np.zeros((64, K), np.uint16); A64[:48] = A
    B64 = np.zeros((N, 64), np.uint16); B64[:, :48] = B
    clef.lora_add(x, bf16_dev(A64), bf16_dev(B64), y64)
    assert torch.equal(y48.view(torch.int16), y64.view(torch.int16))


# ------------------------------------------------------------------ invariances

PIECES = [1, 2, 3, 5, 8, 13, 21, 34, 55, 89, 144, 255]


def pieces(M):
    out, a, i = [], 0, 0
    while a < M:
        n = min(PIECES[i % len(PIECES)], M - a)
        out.append((a, a + n))
        a += n
        i += 1
    return out


def test_row_invariance_int8_fp8_lora():
    """600 rows at once are byte-equal to pieces of 1..255 rows."""
    M, N, K = 600, 512, 2048
    x = bf16_dev(S.activation(0, "t/inv/x", M, K))
    w = bf16_dev(S.weight(0, "t/inv/w", N, K))
    b = bf16_dev(S.bias(0, "t/inv/b", N))
    for mode, lin in (("int8_h128", clef.w8a8_linear), ("fp8", clef.fp8_linear)):
        qx, sx = clef.quant_act(x, mode)
        qw, sw = clef.quant_act(w, mode)
        whole = lin(qx, sx, qw, sw, b)
        part = torch.empty_like(whole)
        for a, c in pieces(M):
            lin(qx[a:c], sx[a:c], qw, sw, b, y=part[a:c])
        assert torch.equal(whole.view(torch.int16), part.view(torch.int16)), mode
    A, B = S.lora_pair(0, "t/inv/l", 256, K, N)
    A, B = bf16_dev(A), bf16_dev(B)
    y0 = bf16_dev(S.normal_bf16(0, "t/inv/y", (M, N)))
    whole = y0.clone()
    clef.lora_add(x, A, B, whole)
    part = y0.clone()
    for a, c in pieces(M):
        clef.lora_add(x[a:c], A, B, part[a:c])
    assert torch.equal(whole.view(torch.int16), part.view(torch.int16)), "lora"


def _same_rows(whole, part, what):
    assert torch.equal(whole.view(torch.int16) if whole.dtype == torch.bfloat16 else whole,
                       part.view(torch.int16) if part.dtype == torch.bfloat16 else part), what


def test_row_invariance_other_kernels():
    """The rest of the path: the quantizer (all modes), the fused gate/up SwiGLU
    (INT8, FP8), the LoRA gate/up + SwiGLU call and the stacked LoRA shrink and
    expand, 600 rows at once against pieces of 1..255 rows."""
    M, N, K, r = 600, 256, 1024, 64
    x = bf16_dev(S.activation(0, "t/inv2/x", M, K))
    for mode in ("int8_h128", "fp8", "fp8_h128"):
        q, sc = clef.quant_act(x, mode)
        qp, sp = torch.empty_like(q), torch.empty_like(sc)
        for a, c in pieces(M):
            clef.quant_act(x[a:c], mode, q=qp[a:c], scale=sp[a:c])
        assert torch.equal(q, qp) and torch.equal(sc, sp), mode
    w = bf16_dev(S.weight(0, "t/inv2/w", 2 * N, K))
    b = bf16_dev(S.bias(0, "t/inv2/b", 2 * N))
    for mode, gu in (("int8_h128", clef.w8a8_gateup_swiglu), ("fp8", clef.fp8_gateup_swiglu)):
        qx, sx = clef.quant_act(x, mode)
        qw, sw = clef.quant_act(w, mode)
        whole = gu(qx, sx, qw, sw, b)
        part = torch.empty_like(whole)
        for a, c in pieces(M):
            gu(qx[a:c], sx[a:c], qw, sw, b, h=part[a:c])
        _same_rows(whole, part, mode + " gate/up")
    Ag, Bg = (bf16_dev(v) for v in S.lora_pair(0, "t/inv2/g", r, K, N))
    Au, Bu = (bf16_dev(v) for v in S.lora_pair(0, "t/inv2/u", r, K, N))
    ygu = bf16_dev(S.normal_bf16(0, "t/inv2/ygu", (M, 2 * N)))
    whole = clef.lora_gateup_swiglu(x, Ag, Bg, Au, Bu, ygu)
    part = torch.empty_like(whole)
    for a, c in pieces(M):
        clef.lora_gateup_swiglu(x[a:c], Ag, Bg, Au, Bu, ygu[a:c], h=part[a:c])
    _same_rows(whole, part, "lora gate/up")
    A_cat = torch.cat([Ag, Au], dim=0)
    t_whole = clef.lora_shrink(x, A_cat)
    t_part = torch.empty_like(t_whole)
    for a, c in pieces(M):
        clef.lora_shrink(x[a:c], A_cat, t=t_part[a:c])
    _same_rows(t_whole, t_part, "lora shrink")
    y0 = bf16_dev(S.normal_bf16(0, "t/inv2/y", (M, N)))
    y_whole, y_part = y0.clone(), y0.clone()
    clef.lora_expand_add(t_whole[:, r:], Bu, y_whole)
    for a, c in pieces(M):
        clef.lora_expand_add(t_whole[a:c, r:], Bu, y_part[a:c])
    _same_rows(y_whole, y_part, "lora expand")


def test_row_invariance_with_stream_k():
    """1,502 rows of the down projection at once split their last 44 tiles
    across all SMs (stream-K); pieces of 1..255 rows never split; the bytes
    agree row for row."""
    M, N, K = 1502, 5120, 17408
    rng = np.random.default_rng(21)
    qx = dev(rng.integers(-127, 128, (M, K)).astype(np.int8))
    qw = dev(rng.integers(-127, 128, (N, K)).astype(np.int8))
    sx = torch.tensor(rng.random(M, dtype=np.float32) * 1e-3, device="cuda")
    sw = torch.tensor(rng.random(N, dtype=np.float32) * 1e-3, device="cuda")
    b = torch.tensor(rng.standard_normal(N, dtype=np.float32), device="cuda").to(torch.bfloat16)
    ws = torch.zeros(clef.gemm_workspace_bytes(), dtype=torch.uint8, device="cuda")
    clef.bind_workspace(ws)
    try:
        whole = clef.w8a8_linear(qx, sx, qw, sw, b)
        part = torch.empty_like(whole)
        for a, c in pieces(M):
            clef.w8a8_linear(qx[a:c], sx[a:c], qw, sw, b, y=part[a:c])
    finally:
        clef.bind_workspace(None)
    _same_rows(whole, part, "int8 stream-K")


def test_two_streams_and_repeats_are_deterministic():
    M, N, K = 1024, 2048, 4096
    x = bf16_dev(S.activation(0, "t/det/x", M, K))
    w = bf16_dev(S.weight(0, "t/det/w", N, K))
    qx, sx = clef.quant_act(x)
    qw, sw = clef.quant_act(w)
    ref = clef.w8a8_linear(qx, sx, qw, sw)
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    torch.cuda.synchronize()
    outs = []
    for s in (s1, s2, s1, s2):
        with torch.cuda.stream(s):
            outs.append(clef.w8a8_linear(qx, sx, qw, sw))
    torch.cuda.synchronize()
    for o in outs:
        assert torch.equal(o.view(torch.int16), ref.view(torch.int16))


def test_empty_calls_are_noops():
    z8 = torch.empty((0, 256), dtype=torch.int8, device="cuda")
    w8 = torch.zeros((64, 256), dtype=torch.int8, device="cuda")
    s0 = torch.empty((0,), dtype=torch.float32, device="cuda")
    sw = torch.ones((64,), dtype=torch.float32, device="cuda")
    y = clef.w8a8_linear(z8, s0, w8, sw)
    assert y.shape == (0, 64)
