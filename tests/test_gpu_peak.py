"""The tensor-core rate microbenchmarks behind the roofline denominators:
each route runs, reports no device error, and lands in a plausible range for
a 152-SM GB300 (the bf16 route near the measured cuBLAS bf16 rate, e4m3 at
roughly twice it, the legacy integer route far below both)."""
import pytest
import torch

import w8a8_quantized_projections_gb300 as clef

pytestmark = pytest.mark.gpu


def test_mma_peaks_plausible():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    bf16 = clef.mma_peak("bf16", 50_000)
    e4m3 = clef.mma_peak("e4m3", 50_000)
    s8 = clef.mma_peak("s8_mma_sync", 2_000)
    assert clef.poll_status() == 0
    assert 500 < bf16 < 3000, bf16
    assert 1.5 * bf16 < e4m3 < 2.5 * bf16, (bf16, e4m3)
    assert 1 < s8 < bf16, (s8, bf16)
