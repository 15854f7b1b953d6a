"""Pins of the CPU oracle against facts that do not come from the oracle itself.

Each check is chosen so that a plausible slip in the oracle (a dropped term, a
wrong sign or index, a transposed operand, a wrong rounding rule) fails it:
closed forms of the Hadamard transform, an independently built Sylvester
matrix, the rotation invariance of the projection, the quantisation error
bound, brute-force nearest-value search for e4m3, library routines (numpy
integer matmul, torch's bf16 / float8_e4m3fn casts and silu) on the cases
where they define the same value, and the LoRA closed form.
"""
import math
import struct
from fractions import Fraction

import numpy as np
import pytest
import torch

import clef_synth as S

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


def f32_bits(f):
    return struct.unpack("<I", struct.pack("<f", f))[0]


def sylvester(n=128):
    """H[i][j] = (-1)^popcount(i & j) / sqrt(n), built from its closed form."""
    i = np.arange(n)
    pc = np.vectorize(lambda v: bin(v).count("1"))(i[:, None] & i[None, :])
    return np.where(pc % 2 == 0, 1.0, -1.0) / math.sqrt(n)


def bf16_ulp(v):
    """Spacing of bf16 at |v| (floored at the smallest normal)."""
    a = np.maximum(np.abs(np.asarray(v, np.float64)), 2.0 ** -126)
    return 2.0 ** (np.floor(np.log2(a)) - 7)


def rot_f64(x_bits):
    """Exact block-128 rotation of bf16 rows, by the fp64 Sylvester matrix."""
    x = S.bf16_bits_to_f64(x_bits)
    M, K = x.shape
    H = sylvester()
    return (x.reshape(M, K // 128, 128) @ H).reshape(M, K)


# ------------------------------------------------------------------ bf16

def test_bf16_rounding_matches_torch(orc):
    rng = np.random.default_rng(1)
    vals = np.concatenate([
        rng.standard_normal(2000).astype(np.float32) * 10.0 ** rng.integers(-8, 8, 2000),
        # exact ties: low half 0x8000 with both parities of the kept half
        (np.arange(1000, dtype=np.uint32) * 0x10000 + 0x3F808000).view(np.float32),
    ]).astype(np.float32)
    want = torch.from_numpy(vals).to(torch.bfloat16).view(torch.int16).numpy().astype(np.uint16)
    got = np.array([orc.f32_to_bf16(float(v)) for v in vals], np.uint16)
    assert np.array_equal(got, want)


def test_f64_to_bf16_is_nearest_even(orc):
    rng = np.random.default_rng(2)
    for d in list(rng.standard_normal(300) * 3.0) + [1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8, -2.5]:
        b = orc.f64_to_bf16(float(d))
        got = Fraction(orc.bf16_to_f32(b))
        # neighbours of the result, all bf16 values; the result must be nearest
        lo = Fraction(orc.bf16_to_f32((b - 1) & 0xFFFF))
        hi = Fraction(orc.bf16_to_f32((b + 1) & 0xFFFF))
        exact = Fraction(float(d))
        assert abs(got - exact) <= abs(lo - exact) and abs(got - exact) <= abs(hi - exact)
        if abs(got - exact) in (abs(lo - exact), abs(hi - exact)) and got != exact:
            assert b % 2 == 0  # tie goes to the even mantissa


# ------------------------------------------------------------------ rotation

def test_normalisation_constant_bits(orc):
    one = np.zeros(128, np.float32)
    one[0] = 1.0
    v = orc.wht128_f32(one)
    assert f32_bits(float(v[0])) == 0x3DB504F3


@pytest.mark.parametrize("j", [0, 1, 5, 64, 77, 127])
def test_one_hot_closed_form(orc, j):
    e = np.zeros(128, np.float32)
    e[j] = 1.0
    v = orc.wht128_f32(e)
    c = np.float32(1.0 / math.sqrt(128.0))
    signs = np.array([1.0 if bin(i & j).count("1") % 2 == 0 else -1.0 for i in range(128)], np.float32)
    assert np.array_equal(v, signs * c)


def test_all_ones_closed_form(orc):
    v = orc.wht128_f32(np.ones(128, np.float32))
    assert v[0] == np.float32(128.0) * np.float32(1.0 / math.sqrt(128.0))
    assert np.all(v[1:] == 0.0)


def test_f64_transform_equals_sylvester_matrix(orc):
    rng = np.random.default_rng(3)
    H = sylvester()
    for _ in range(5):
        x = rng.standard_normal(128)
        assert np.allclose(orc.wht128_f64(x), H @ x, rtol=0, atol=1e-13)


def test_orthonormal_and_involutive(orc):
    cols = np.stack([orc.wht128_f64(np.eye(128)[j]) for j in range(128)], axis=1)
    assert np.allclose(cols @ cols.T, np.eye(128), atol=1e-14)
    rng = np.random.default_rng(4)
    x = rng.standard_normal(128)
    assert np.allclose(orc.wht128_f64(orc.wht128_f64(x)), x, atol=1e-14)
    # fp32: rotating twice returns bf16 inputs within the rounding of 16 ops
    xb = S.f64_to_bf16_bits(rng.standard_normal(128))
    xf = S.bf16_bits_to_f64(xb).astype(np.float32)
    back = orc.wht128_f32(orc.wht128_f32(xf)).astype(np.float64)
    assert np.max(np.abs(back - xf)) <= 2.0 ** -18 * np.linalg.norm(xf)


def test_rotate_rows_against_exact(orc):
    x = S.activation(0, "pin/rot", 5, 384)
    got = orc.rotate_rows(x).astype(np.float64)
    ref = rot_f64(x)
    # 7 rounded stages + 1 rounded multiply: |err| <= 8 u * sum |x| per block
    xa = np.abs(S.bf16_bits_to_f64(x)).reshape(5, 3, 128).sum(-1)
    bound = np.repeat(8 * 2.0 ** -24 * xa / math.sqrt(128) * 2, 128, axis=1)
    assert np.all(np.abs(got - ref) <= bound + 1e-30)


def test_rotation_invariance_of_projection(orc):
    x = S.bf16_bits_to_f64(S.activation(0, "pin/inv_x", 4, 256))
    w = S.bf16_bits_to_f64(S.weight(0, "pin/inv_w", 6, 256))
    rot = lambda a: np.stack([np.concatenate([orc.wht128_f64(r[b:b + 128]) for b in range(0, 256, 128)]) for r in a])
    lhs = x @ w.T
    rhs = rot(x) @ rot(w).T
    assert np.allclose(lhs, rhs, rtol=1e-12, atol=1e-12 * np.abs(lhs).max())


# ------------------------------------------------------------------ INT8 quantiser

def test_int8_quant_error_bound_and_amax_code(orc):
    x = S.activation(0, "pin/q8", 7, 512)
    q, s = orc.quant_int8_h128(x)
    v = orc.rotate_rows(x).astype(np.float64)
    deq = q.astype(np.float64) * s[:, None].astype(np.float64)
    assert np.all(np.abs(v - deq) <= s[:, None] / 2 * (1 + 2.0 ** -20))
    assert np.all(np.abs(q).max(axis=1) == 127)
    assert q.min() >= -127
    # the amax element carries code +-127 with its own sign
    idx = np.abs(v).argmax(axis=1)
    assert np.all(q[np.arange(7), idx] == np.sign(v[np.arange(7), idx]) * 127)
    # scale is amax / 127 with amax the exact max of the rotated row
    amax = np.abs(orc.rotate_rows(x)).max(axis=1)
    assert np.array_equal(s, (amax / np.float32(127.0)).astype(np.float32))


def test_int8_quant_one_hot_and_zero_rows(orc):
    x = np.zeros((2, 256), np.uint16)
    x[0, 3] = S.f64_to_bf16_bits(np.array([-1.5]))[0]
    q, s = orc.quant_int8_h128(x)
    signs = np.array([1 if bin(i & 3).count("1") % 2 == 0 else -1 for i in range(128)])
    assert np.array_equal(q[0, :128], -127 * signs)
    assert np.all(q[0, 128:] == 0)
    c = np.float32(1.0 / math.sqrt(128.0))
    assert s[0] == np.float32(np.float32(1.5) * c) / np.float32(127.0)
    assert s[1] == 0.0 and np.all(q[1] == 0)


def test_int8_codes_are_rint_of_scaled_values(orc):
    """Codes are numpy's round-half-even rint of fp32(v * (127/amax)), on the
    oracle's rotated values (the rotation is pinned above).  Random rows
    almost never land on an exact half; the next test builds such cases."""
    x = S.activation(0, "pin/rint", 4, 256)
    q, _ = orc.quant_int8_h128(x)
    v = orc.rotate_rows(x)
    amax = np.abs(v).max(1, keepdims=True)
    r = (np.float32(127.0) / amax).astype(np.float32)
    want = np.clip(np.rint((v * r).astype(np.float32)), -127, 127).astype(np.int8)
    assert np.array_equal(q, want)
    # np.rint itself rounds ties to even (the rule the codes follow)
    assert np.array_equal(np.rint(np.array([0.5, 1.5, 2.5, -0.5, -2.5])), [0, 2, 2, -0, -2])


def test_int8_code_ties_round_to_even(orc):
    """Exact halves: a row of 0.5s rotates to v = fp32(64 c) at index 0 and
    zeros elsewhere; static scales s found next to v / target give
    fp32(v * fp32(1/s)) equal to target, an exact half with an even integer
    below it.  Round-half-even keeps that integer (either sign), so a
    round-half-up or half-away rule fails here."""
    c = np.float32(1.0 / math.sqrt(128.0))
    v = np.float32(np.float32(64.0) * c)
    x = np.stack([S.f64_to_bf16_bits(np.full(128, 0.5)), S.f64_to_bf16_bits(np.full(128, -0.5))])
    rot = orc.rotate_rows(x)
    assert rot[0, 0] == v and rot[1, 0] == -v and not rot[:, 1:].any()
    found = []
    for target in (0.5, 2.5, 12.5, 62.5, 100.5, 126.5):
        s0 = np.float32(v / np.float32(target))
        for d in range(-64, 65):
            sc = (np.array([s0], np.float32).view(np.int32) + d).view(np.float32)[0]
            if np.float32(v * (np.float32(1.0) / sc)) == np.float32(target):
                found.append((sc, target))
                break
    assert len(found) >= 3, found
    for sc, target in found:
        q, _ = orc.quant_static(x, float(sc), "int8_h128")
        even = int(target - 0.5)
        assert even % 2 == 0
        assert q[0, 0] == even and q[1, 0] == -even, (target, q[:, 0])
        assert not q[:, 1:].any()


def test_static_int8_codes_are_clamped_rint(orc):
    """Static scale: codes are numpy's rint of fp32(v * fp32(1/s)) on the
    (pinned) rotated values, clamped to [-127, 127] (a static scale lets
    values overflow the range, unlike the per-token one); every row's scale
    is s.  s = 2^-4 makes v * r exact, s = 0.037 exercises a rounded r."""
    x = S.activation(0, "pin/static8", 5, 256)
    v = orc.rotate_rows(x)
    for sc in (0.0625, 0.037):
        q, sout = orc.quant_static(x, sc, "int8_h128")
        r = np.float32(1.0) / np.float32(sc)
        want = np.clip(np.rint((v * r).astype(np.float32)), -127, 127).astype(np.int8)
        assert np.array_equal(q, want) and np.all(sout == np.float32(sc))
        assert (np.abs(v * r) > 127.5).any(), "some values saturate"
        assert q.min() == -127 and q.max() == 127


def test_static_fp8_codes_match_the_encoder_and_saturate(orc):
    """Static FP8: each code is the (pinned) e4m3 encoding of fp32(v * fp32(1/s)),
    unrotated and rotated; values beyond 448 * s saturate to +-448; with a
    power-of-two s the codes equal torch's float8 cast of v / s."""
    x = S.activation(0, "pin/static8f", 4, 256)
    for mode, v in (("fp8", S.bf16_bits_to_f64(x).astype(np.float32)), ("fp8_h128", orc.rotate_rows(x))):
        for sc in (2.0 ** -7, 0.0123):
            q, sout = orc.quant_static(x, sc, mode)
            t = (v * (np.float32(1.0) / np.float32(sc))).astype(np.float32)
            want = np.array([orc.e4m3_encode(float(f)) for f in t.ravel()], np.uint8).reshape(t.shape)
            assert np.array_equal(q, want) and np.all(sout == np.float32(sc))
            big = np.abs(t) >= 448
            assert big.any() and np.all((q[big] & 0x7F) == 0x7E)
            if sc == 2.0 ** -7:
                ref = torch.from_numpy(np.clip(t, -448, 448)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
                assert np.array_equal(q, ref)


# ------------------------------------------------------------------ e4m3

def _finite_codes():
    return [c for c in range(256) if (c & 0x7F) != 0x7F]


def test_e4m3_decode_table(orc):
    known = {0x00: 0.0, 0x01: 2.0 ** -9, 0x07: 7 * 2.0 ** -9, 0x08: 2.0 ** -6, 0x38: 1.0,
             0x39: 1.125, 0x7E: 448.0, 0xFE: -448.0, 0xB8: -1.0, 0x40: 2.0}
    for c, v in known.items():
        assert orc.e4m3_decode(c) == v
    assert math.isnan(orc.e4m3_decode(0x7F)) and math.isnan(orc.e4m3_decode(0xFF))
    pos = [orc.e4m3_decode(c) for c in range(0x7F)]
    assert all(a < b for a, b in zip(pos, pos[1:]))  # strictly increasing
    assert len(set(pos)) == 127                        # 126 positive finite + zero


def test_e4m3_encode_brute_force(orc):
    vals = [(c, orc.e4m3_decode(c)) for c in _finite_codes()]

    def nearest(f):
        if abs(f) >= 448.0:
            return 0x7E | (0x80 if f < 0 else 0)
        best = None
        for c, v in vals:
            if (c & 0x80) != (0x80 if math.copysign(1.0, f) < 0 else 0):
                continue
            d = abs(Fraction(v) - Fraction(f))
            key = (d, c & 1)  # ties: even mantissa (code LSB 0)
            if best is None or key < best[0]:
                best = (key, c)
        return best[1]

    pts = []
    pos = [orc.e4m3_decode(c) for c in range(0x7F)]
    for a, b in zip(pos, pos[1:]):
        mid = np.float32((a + b) / 2)
        pts += [mid, np.nextafter(mid, np.float32(0)), np.nextafter(mid, np.float32(1e9))]
    rng = np.random.default_rng(5)
    pts += list((rng.standard_normal(400) * 100).astype(np.float32))
    pts += list((rng.standard_normal(100) * 0.01).astype(np.float32))
    pts += [np.float32(v) for v in (447.9, 448.0, 463.9, 464.0, 480.0, 1e6, 2.0 ** -10, 2.0 ** -11, 0.0)]
    for p in pts:
        for f in (float(p), -float(p)):
            assert orc.e4m3_encode(f) == nearest(f), f


def test_e4m3_round_trip_and_torch(orc):
    for c in _finite_codes():
        assert orc.e4m3_encode(orc.e4m3_decode(c)) == c
    rng = np.random.default_rng(6)
    v = (rng.standard_normal(3000) * 60).astype(np.float32)
    v = v[np.abs(v) <= 448]
    want = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = np.array([orc.e4m3_encode(float(f)) for f in v], np.uint8)
    assert np.array_equal(got, want)


def test_fp8_quant_bound(orc):
    x = S.activation(0, "pin/q_fp8", 6, 320)
    for rotate in (False, True):
        if rotate and 320 % 128:
            continue
        q, s = orc.quant_fp8(x, rotate=rotate)
        v = S.bf16_bits_to_f64(x)
        assert np.array_equal(s, (np.abs(v).max(1).astype(np.float32) / np.float32(448)).astype(np.float32))
        deq = np.vectorize(orc.e4m3_decode)(q) * s[:, None]
        # e4m3 relative step 2^-3 (half of it after rounding), plus the subnormal floor
        err = np.abs(deq - v)
        assert np.all(err <= np.abs(v) * 2.0 ** -4 * 1.001 + s[:, None] * 2.0 ** -10 * 1.001)
        assert np.all(np.abs(np.vectorize(orc.e4m3_decode)(q)).max(1) == 448.0)
    xr = S.activation(0, "pin/q_fp8r", 3, 256)
    q, s = orc.quant_fp8(xr, rotate=True)
    v = orc.rotate_rows(xr).astype(np.float64)
    deq = np.vectorize(orc.e4m3_decode)(q) * s[:, None]
    assert np.all(np.abs(deq - v) <= np.abs(v) * 2.0 ** -4 * 1.001 + s[:, None] * 2.0 ** -10 * 1.001)


# ------------------------------------------------------------------ INT8 GEMM

def test_int8_gemm_against_numpy_and_bruteforce(orc):
    rng = np.random.default_rng(7)
    for (M, N, K) in [(1, 1, 128), (5, 7, 256), (8, 3, 384)]:
        a = rng.integers(-127, 128, (M, K), dtype=np.int64).astype(np.int8)
        b = rng.integers(-127, 128, (N, K), dtype=np.int64).astype(np.int8)
        got = orc.int8_gemm_acc(a, b)
        assert np.array_equal(got, a.astype(np.int64) @ b.astype(np.int64).T)
    a = rng.integers(-127, 128, (2, 128)).astype(np.int8)
    b = rng.integers(-127, 128, (3, 128)).astype(np.int8)
    brute = [[sum(int(a[i, k]) * int(b[j, k]) for k in range(128)) for j in range(3)] for i in range(2)]
    assert orc.int8_gemm_acc(a, b).tolist() == brute


def test_int8_gemm_extremes(orc):
    K = 17408
    a = np.full((1, K), 127, np.int8)
    assert orc.int8_gemm_acc(a, a)[0, 0] == 16129 * K == 280773632
    assert orc.int8_gemm_acc(a, -a)[0, 0] == -280773632


def test_int8_linear_approximates_unquantised_projection(orc):
    """The full INT8 path (rotate, quantise both sides, GEMM, epilogue) lands
    within the derived quantisation bound of the fp64 projection x W^T + b."""
    M, N, K = 6, 40, 512
    x = S.activation(0, "pin/lin_x", M, K)
    w = S.weight(0, "pin/lin_w", N, K)
    b = S.bias(0, "pin/lin_b", N)
    qx, sx = orc.quant_int8_h128(x)
    qw, sw = orc.quant_int8_h128(w)
    y = S.bf16_bits_to_f64(orc.int8_linear(qx, sx, qw, sw, b))
    xf, wf, bf = (S.bf16_bits_to_f64(t) for t in (x, w, b))
    ref = xf @ wf.T + bf
    vx, vw = rot_f64(x), rot_f64(w)
    sx6, sw6 = sx.astype(np.float64)[:, None], sw.astype(np.float64)[:, None]
    bound = (np.abs(vx) @ (np.ones((N, K)) * sw6 / 2).T + (sx6 / 2) @ np.abs(vw).sum(1)[None, :]
             + K * sx6 * sw6.T / 4)
    bound = bound + 1e-4 * np.abs(ref) + bf16_ulp(ref)
    assert np.all(np.abs(y - ref) <= bound)
    # and the scales matter: dropping the weight scale breaks the bound
    y_bad = S.bf16_bits_to_f64(orc.int8_linear(qx, sx, qw, np.ones_like(sw), b))
    assert not np.all(np.abs(y_bad - ref) <= bound)


def test_int8_linear_exact_cases(orc):
    # s = sw = 1, no bias: y = bf16(acc) (torch's cast as the rounding routine)
    rng = np.random.default_rng(8)
    a = rng.integers(-127, 128, (3, 256)).astype(np.int8)
    b = rng.integers(-127, 128, (5, 256)).astype(np.int8)
    y = orc.int8_linear(a, np.ones(3, np.float32), b, np.ones(5, np.float32))
    acc = torch.from_numpy(a.astype(np.int64) @ b.astype(np.int64).T).float()
    assert np.array_equal(y, acc.to(torch.bfloat16).view(torch.int16).numpy().astype(np.uint16))
    # power-of-two scales are exact: y = bf16(acc * 2^-10 + bias)
    bias = S.bias(0, "pin/b", 5)
    y2 = orc.int8_linear(a, np.full(3, 2.0 ** -5, np.float32), b, np.full(5, 2.0 ** -5, np.float32), bias)
    want = (torch.from_numpy(a.astype(np.int64) @ b.astype(np.int64).T).double() * 2.0 ** -10
            + torch.from_numpy(S.bf16_bits_to_f64(bias)))
    # acc*2^-10 is exact in fp32 and the single fp32 add then bf16 equals torch's
    # fp32 add then cast
    want = want.float().to(torch.bfloat16).view(torch.int16).numpy().astype(np.uint16)
    assert np.array_equal(y2, want)
    # a bias as large as the scaled products, one value per output channel:
    # dropping it, or indexing it by row, changes the outputs
    big = S.f64_to_bf16_bits(np.array([3.0, -5.0, 0.5, 7.0, -1.25]))
    y3 = orc.int8_linear(a, np.full(3, 2.0 ** -8, np.float32), b, np.full(5, 2.0 ** -8, np.float32), big)
    want3 = (torch.from_numpy(a.astype(np.int64) @ b.astype(np.int64).T).double() * 2.0 ** -16
             + torch.tensor([3.0, -5.0, 0.5, 7.0, -1.25], dtype=torch.float64))
    want3 = want3.float().to(torch.bfloat16).view(torch.int16).numpy().astype(np.uint16)
    assert np.array_equal(y3, want3)
    no_bias = orc.int8_linear(a, np.full(3, 2.0 ** -8, np.float32), b, np.full(5, 2.0 ** -8, np.float32))
    assert (y3 != no_bias).all()


# ------------------------------------------------------------------ SwiGLU

def test_silu_identities_and_torch(orc):
    assert orc.swiglu_f32(0.0, 1.0) == 0.0
    rng = np.random.default_rng(9)
    g = (rng.standard_normal(500) * 6).astype(np.float32)
    for gi in g[:100]:
        lhs = orc.swiglu_f32(float(gi), 1.0) - orc.swiglu_f32(float(-gi), 1.0)
        assert abs(lhs - float(gi)) <= 4 * abs(float(gi)) * 2.0 ** -23 + 1e-30
    ref64 = g.astype(np.float64) / (1.0 + np.exp(-g.astype(np.float64)))
    got = np.array([orc.swiglu_f32(float(v), 1.0) for v in g], np.float64)
    assert np.all(np.abs(got - ref64) <= 3 * np.abs(ref64) * 2.0 ** -24 + 1e-37)
    tor = torch.nn.functional.silu(torch.from_numpy(g)).double().numpy()
    assert np.all(np.abs(got - tor) <= 4 * np.abs(ref64) * 2.0 ** -24 + 1e-37)
    assert orc.swiglu_f32(60.0, 3.0) == 180.0
    assert orc.swiglu_f32(-200.0, 3.0) == 0.0 or abs(orc.swiglu_f32(-200.0, 3.0)) < 1e-80


def test_gateup_packing_order_and_formula(orc):
    # qx = e_0 (code 1), scales 1: g = qw_gate[n][0], u = qw_up[n][0]
    N, K = 4, 128
    qx = np.zeros((1, K), np.int8)
    qx[0, 0] = 1
    qw = np.zeros((2 * N, K), np.int8)
    gate = np.array([3, -2, 0, 7])
    up = np.array([5, 1, 9, -4])
    qw[:N, 0] = gate
    qw[N:, 0] = up
    h = S.bf16_bits_to_f64(orc.int8_gateup_swiglu(qx, np.ones(1, np.float32), qw, np.ones(2 * N, np.float32)))
    ref = gate / (1 + np.exp(-gate)) * up
    assert np.all(np.abs(h[0] - ref) <= bf16_ulp(ref))
    swapped = up / (1 + np.exp(-up)) * gate
    assert not np.allclose(h[0], swapped)


def test_unfused_swiglu_close_to_fused(orc):
    M, N, K = 4, 32, 256
    x = S.activation(0, "pin/gu_x", M, K)
    w = S.weight(0, "pin/gu_w", 2 * N, K)
    qx, sx = orc.quant_int8_h128(x)
    qw, sw = orc.quant_int8_h128(w)
    fused = S.bf16_bits_to_f64(orc.int8_gateup_swiglu(qx, sx, qw, sw))
    y_gu = orc.int8_linear(qx, sx, qw, sw)
    unfused = S.bf16_bits_to_f64(orc.swiglu_bf16(y_gu))
    g = S.bf16_bits_to_f64(y_gu[:, :N])
    u = S.bf16_bits_to_f64(y_gu[:, N:])
    # two extra bf16 roundings of g and u: |d h| <= |dsilu|*|dg|*|u| + |silu|*|du| + 2 ulp
    bound = (1.1 * np.abs(u) * bf16_ulp(g) + np.abs(g) * bf16_ulp(u) + 2 * bf16_ulp(fused))
    assert np.all(np.abs(fused - unfused) <= bound)


# ------------------------------------------------------------------ FP8 GEMM

def test_fp8_linear_exact_sum(orc):
    rng = np.random.default_rng(10)
    M, N, K = 3, 4, 64
    fin = np.array(_finite_codes(), np.uint8)
    qx = rng.choice(fin, (M, K)).astype(np.uint8)
    qw = rng.choice(fin, (N, K)).astype(np.uint8)
    sx = (rng.random(M) + 0.5).astype(np.float32)
    sw = (rng.random(N) + 0.5).astype(np.float32)
    bias = S.bias(0, "pin/fp8b", N)
    y = orc.fp8_linear(qx, sx, qw, sw, bias)
    for m in range(M):
        for n in range(N):
            exact = sum(Fraction(orc.e4m3_decode(int(qx[m, k]))) * Fraction(orc.e4m3_decode(int(qw[n, k])))
                        for k in range(K))
            acc = np.float32(float(exact))  # float(Fraction) is correctly rounded to fp64 first
            v = np.float32(np.float32(acc * sx[m]) * sw[n])
            v = np.float32(v + np.float32(orc.bf16_to_f32(int(bias[n]))))
            assert y[m, n] == orc.f32_to_bf16(float(v))
    # scales of 2^-40 shrink every product below 2^-15 of the bias, so the output is
    # the per-channel bias itself (a dropped or row-indexed bias fails)
    big = np.array([3.0, -5.0, 0.5, 7.0])
    y2 = orc.fp8_linear(qx, np.full(M, 2.0 ** -40, np.float32), qw, np.full(N, 2.0 ** -40, np.float32),
                        S.f64_to_bf16_bits(big))
    assert np.array_equal(S.bf16_bits_to_f64(y2), np.tile(big, (M, 1)))


def test_fp8_linear_approximates_projection(orc):
    M, N, K = 5, 24, 512
    x = S.activation(0, "pin/f8_x", M, K)
    w = S.weight(0, "pin/f8_w", N, K)
    qx, sx = orc.quant_fp8(x)
    qw, sw = orc.quant_fp8(w)
    y = S.bf16_bits_to_f64(orc.fp8_linear(qx, sx, qw, sw))
    ref = S.bf16_bits_to_f64(x) @ S.bf16_bits_to_f64(w).T
    rms = np.sqrt(np.mean(ref ** 2))
    assert np.sqrt(np.mean((y - ref) ** 2)) < 0.08 * rms


# ------------------------------------------------------------------ LoRA

def test_lora_identity_closed_form(orc):
    M, K, r = 5, 128, 64
    x = S.activation(0, "pin/lx", M, K)
    A = np.zeros((r, K), np.uint16)
    A[np.arange(r), np.arange(r)] = 0x3F80  # bf16 1.0
    B = np.zeros((r, r), np.uint16)
    B[np.arange(r), np.arange(r)] = 0x3F80
    y = S.normal_bf16(0, "pin/ly", (M, r))
    out = orc.lora_add(x, A, B, y)
    want = torch.from_numpy(S.bf16_bits_to_f64(y) + S.bf16_bits_to_f64(x[:, :r])).float()
    # y + x is one fp32 add of two bf16 values (exact), then one bf16 rounding
    want = want.to(torch.bfloat16).view(torch.int16).numpy().astype(np.uint16)
    assert np.array_equal(out, want)


def test_lora_zero_padding_is_exact(orc):
    M, K, N, r = 6, 256, 40, 48
    x = S.activation(0, "pin/pad_x", M, K)
    A, B = S.lora_pair(0, "pin/pad", r, K, N)
    y = S.normal_bf16(0, "pin/pad_y", (M, N))
    t48 = orc.lora_t(x, A, r_pad=48)
    t64 = orc.lora_t(x, A, r_pad=64)
    assert np.array_equal(t64[:, :48], t48) and np.all(t64[:, 48:] == 0)
    assert np.array_equal(orc.lora_y(t48, B, y), orc.lora_y(t64, B, y))


def test_lora_against_fp64_and_row_invariance(orc):
    M, K, N, r = 40, 256, 24, 64
    x = S.activation(0, "pin/li_x", M, K)
    A, B = S.lora_pair(0, "pin/li", r, K, N)
    y = S.normal_bf16(0, "pin/li_y", (M, N))
    t = orc.lora_t(x, A)
    exact_t = S.bf16_bits_to_f64(x) @ S.bf16_bits_to_f64(A).T
    assert np.all(np.abs(S.bf16_bits_to_f64(t) - exact_t) <= bf16_ulp(exact_t) / 2 * 1.0001)
    out = orc.lora_y(t, B, y)
    z = S.bf16_bits_to_f64(t) @ S.bf16_bits_to_f64(B).T + S.bf16_bits_to_f64(y)
    assert np.all(np.abs(S.bf16_bits_to_f64(out) - z) <= bf16_ulp(z) * 0.5001 + 2.0 ** -23 * np.abs(z))
    pieces = np.concatenate([orc.lora_add(x[a:a + 7], A, B, y[a:a + 7]) for a in range(0, M, 7)])
    assert np.array_equal(pieces, orc.lora_add(x, A, B, y))


def test_fp8_gateup_swiglu_matches_linear_halves(orc):
    """The fused FP8 SwiGLU oracle agrees with silu(gate) * up formed from the
    oracle's FP8 linear halves (which round g and u to bf16 first)."""
    M, N, K = 3, 16, 256
    x = S.activation(0, "pin/f8gu_x", M, K)
    w = S.weight(0, "pin/f8gu_w", 2 * N, K)
    qx, sx = orc.quant_fp8(x)
    qw, sw = orc.quant_fp8(w)
    h = S.bf16_bits_to_f64(orc.fp8_gateup_swiglu(qx, sx, qw, sw))
    y = orc.fp8_linear(qx, sx, qw, sw)
    g, u = S.bf16_bits_to_f64(y[:, :N]), S.bf16_bits_to_f64(y[:, N:])
    ref = g / (1 + np.exp(-g)) * u
    bound = 1.1 * np.abs(u) * bf16_ulp(g) + np.abs(g) * bf16_ulp(u) + 2 * bf16_ulp(ref)
    assert np.all(np.abs(h - ref) <= bound)
