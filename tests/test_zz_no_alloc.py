"""clef_lora_add_noalloc: the LoRA add for callers that cannot allocate
device memory (a runtime that owns a fixed memory budget, a plugin inside
another framework's allocator, code that must avoid the synchronisation of
cudaMalloc).  It keeps t in a built-in device array instead of a caller
scratch.  Checked through the C ABI against clef_lora_add, byte for byte, on
two calls in a row (different shapes and data, so the second call runs over
the first call's leftovers) and on the largest accepted size.  Collected
last so that a run stopping at the first failure has run everything else."""
import ctypes as C

import numpy as np
import pytest
import torch

import clef_synth as S
import w8a8_quantized_projections_gb300 as clef
from gpu_util import bf16_dev, bf16_host

pytestmark = pytest.mark.gpu


def run_pair(call, M, K, N, r):
    """clef_lora_add (caller scratch) and clef_lora_add_noalloc on the same
    seeded inputs; returns both outputs as bf16 bits."""
    x = S.activation(call, f"noalloc/{call}/x", M, K)
    A, B = S.lora_pair(call, f"noalloc/{call}", r, K, N)
    y0 = S.normal_bf16(call, f"noalloc/{call}/y", (M, N))
    xd, Ad, Bd = bf16_dev(x), bf16_dev(A), bf16_dev(B)
    t_dev = torch.empty((M, clef.lora_pad(r)), dtype=torch.bfloat16, device="cuda")
    y_ref = bf16_dev(y0)
    clef.lora_add(xd, Ad, Bd, y_ref, t_scratch=t_dev)
    y_na = bf16_dev(y0)
    clef.lora_add_noalloc(xd, Ad, Bd, y_na)
    torch.cuda.synchronize()
    return bf16_host(y_ref), bf16_host(y_na)


def test_noalloc_matches_scratch_entry_point_twice():
    """Both entry points run the same launches (tile widths, order and
    arguments) and differ only in where t lives, so their outputs must be
    byte-equal; any difference would mean stale or misaddressed scratch.  The
    second call has other shapes and data, so it runs over the first call's
    leftovers in the array."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    for call, (M, K, N, r) in enumerate([(300, 2048, 1024, 256), (130, 1024, 264, 48)]):
        ref, got = run_pair(call, M, K, N, r)
        assert np.array_equal(got, ref), f"call {call}: {int((got != ref).sum())} outputs differ"
    assert clef.poll_status() == 0


def test_noalloc_at_its_size_limit():
    """The largest accepted call: M * round_up(r, 64) equal to the array's
    4,194,304 elements (16,384 rows at rank 256), byte-equal to clef_lora_add."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    ref, got = run_pair(2, 16384, 512, 256, 256)
    assert np.array_equal(got, ref), f"{int((got != ref).sum())} outputs differ"
    assert clef.poll_status() == 0


def test_noalloc_rejects_sizes_beyond_its_scratch():
    """Host-side check: 16,385 rows at rank 256 exceed the 4 Mi-element array."""
    L = clef.library()
    p = C.c_void_p(0x10000)
    rc = L.clef_lora_add_noalloc(p, 256, p, p, 16385, 256, 64, 256, p, 64, C.c_void_p(None))
    assert rc == 1
    assert b"exceeds" in L.clef_last_error()
