"""clef_lora_add_noalloc: the LoRA add for callers that cannot allocate
device memory (a runtime that owns a fixed memory budget, a plugin inside
another framework's allocator, code that must avoid the synchronisation of
cudaMalloc).  It keeps t in a built-in device array instead of a caller
scratch.  Checked through the C ABI against clef_lora_add on two calls in a
row (different shapes and data, so the second call runs over the first
call's leftovers), with the tolerance of the LoRA parity tests.  Collected
last so that a run stopping at the first failure has run everything else."""
import ctypes as C

import numpy as np
import pytest
import torch

import clef_synth as S
import w8a8_quantized_projections_gb300 as clef
from gpu_util import bf16_dev, bf16_host, bf16_ulp

pytestmark = pytest.mark.gpu


def tolerance(x, A, B, t, y_ref, K, r_pad):
    """1 ulp of the result, plus t's error bound (1 ulp + 2 gamma_K sum|xA|)
    carried through |B|, plus stage 2's fp32 accumulation bound."""
    gk = (K / 16 + 2) * 2.0 ** -23
    gr = (r_pad / 16 + 2) * 2.0 ** -23
    r = A.shape[0]
    tv = S.bf16_bits_to_f64(t)[:, :r]
    xa = np.abs(S.bf16_bits_to_f64(x)) @ np.abs(S.bf16_bits_to_f64(A)).T
    Bv = np.abs(S.bf16_bits_to_f64(B))
    return (bf16_ulp(S.bf16_bits_to_f64(y_ref)) + (bf16_ulp(tv) + 2 * gk * xa) @ Bv.T
            + 2 * gr * (np.abs(tv) @ Bv.T))


def test_noalloc_matches_scratch_entry_point_twice():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    for call, (M, K, N, r) in enumerate([(300, 2048, 1024, 256), (130, 1024, 264, 48)]):
        x = S.activation(call, f"noalloc/{call}/x", M, K)
        A, B = S.lora_pair(call, f"noalloc/{call}", r, K, N)
        y0 = S.normal_bf16(call, f"noalloc/{call}/y", (M, N))
        xd, Ad, Bd = bf16_dev(x), bf16_dev(A), bf16_dev(B)
        r_pad = clef.lora_pad(r)
        t_dev = torch.empty((M, r_pad), dtype=torch.bfloat16, device="cuda")
        y_ref = bf16_dev(y0)
        clef.lora_add(xd, Ad, Bd, y_ref, t_scratch=t_dev)
        y_na = bf16_dev(y0)
        clef.lora_add_noalloc(xd, Ad, Bd, y_na)
        torch.cuda.synchronize()
        ref, got = bf16_host(y_ref), bf16_host(y_na)
        tol = tolerance(x, A, B, bf16_host(t_dev), ref, K, r_pad)
        d = np.abs(S.bf16_bits_to_f64(got) - S.bf16_bits_to_f64(ref))
        assert np.all(d <= tol), f"call {call}: worst excess {(d - tol).max():.3g}"
    assert clef.poll_status() == 0


def test_noalloc_rejects_sizes_beyond_its_scratch():
    """Host-side check: 16,385 rows at rank 256 exceed the 4 Mi-element array."""
    L = clef.library()
    p = C.c_void_p(0x10000)
    rc = L.clef_lora_add_noalloc(p, 256, p, p, 16385, 256, 64, 256, p, 64, C.c_void_p(None))
    assert rc == 1
    assert b"exceeds" in L.clef_last_error()
