"""The round-trip smoke pass (quantizer, INT8 linear, gate/up SwiGLU, FP8
linear, LoRA add on cuda:0, each against the CPU oracle) runs as a test, so
its tolerances stay the ones the parity tests use."""
import os
import sys

import pytest

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))


@pytest.mark.gpu
def test_smoke_pass():
    import __graft_entry__ as g
    g.smoke()
