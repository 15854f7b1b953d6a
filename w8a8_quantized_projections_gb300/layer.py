"""One decoder layer's quantized projections, run through the C ABI.

``QuantizedLayer`` quantizes the bf16 weights once at set-up with the same
quantizer the activations use (INT8: block-128 rotation and per-output-channel
scales; FP8: per-channel e4m3 from the weights alone, as the "clef-flash-FP8"
model card's Quantization table describes), packs gate and up side by side
(gate rows first, as the "Loading CLEF INT8" usage notes pack them at load),
and preallocates every activation-code, scale, scratch and output buffer so
that a ``step`` launches kernels only.

A step runs, per distinct activation tensor, one quantizer call, then per
projection one GEMM call (gate/up with the fused SwiGLU epilogue).  With
runtime LoRA pairs, every adapted projection adds ``bf16(x A^T) B^T`` after
its GEMM; gate/up is then run as a packed linear (bf16 gate and up), the LoRA
adds land on each half before the nonlinearity, and the unfused SwiGLU kernel
forms h.
"""
from __future__ import annotations

from typing import Dict, Optional, Tuple

import torch

from . import (fp8_gateup_swiglu, fp8_linear, lora_add, lora_pad, quant_act, swiglu_bf16,
               w8a8_gateup_swiglu, w8a8_linear)


class QuantizedLayer:
    def __init__(self, cfg, weights: Dict[str, Tuple[torch.Tensor, Optional[torch.Tensor]]],
                 lora: Optional[Dict[str, Tuple[torch.Tensor, torch.Tensor]]] = None,
                 device="cuda"):
        """weights: projection name -> (W bf16 [rows][K], bias bf16 [rows] or None);
        lora: name (or name + "/gate", name + "/up" for gate/up) -> (A, B)."""
        self.cfg = cfg
        self.M = cfg.M
        self.fp8 = cfg.scheme == "fp8"
        self.mode = "fp8" if self.fp8 else "int8_h128"
        self.lora = lora or {}
        self.w = {}
        for p in cfg.projections:
            W, b = weights[p.name]
            qw, sw = quant_act(W, self.mode)
            self.w[p.name] = (qw, sw, b)
        torch.cuda.synchronize()
        M = self.M
        code = torch.uint8 if self.fp8 else torch.int8
        self.q = {}
        for name, K in cfg.activations():
            self.q[name] = (torch.empty((M, K), dtype=code, device=device),
                            torch.empty((M,), dtype=torch.float32, device=device))
        self.out = {}
        for p in cfg.projections:
            if p.kind == "gateup":
                self.out[p.name] = torch.empty((M, p.N), dtype=torch.bfloat16, device=device)
                if self.lora:
                    self.out[p.name + "/packed"] = torch.empty((M, 2 * p.N), dtype=torch.bfloat16,
                                                               device=device)
            else:
                self.out[p.name] = torch.empty((M, p.N), dtype=torch.bfloat16, device=device)
            if p.chained:
                self.q[p.act] = (torch.empty((M, p.K), dtype=code, device=device),
                                 torch.empty((M,), dtype=torch.float32, device=device))
        # one dense LoRA scratch [M][r_pad] per padded rank in use
        self.t = {}
        for A, _ in self.lora.values():
            r_pad = lora_pad(A.shape[0])
            if r_pad not in self.t:
                self.t[r_pad] = torch.empty((M, r_pad), dtype=torch.bfloat16, device=device)

    def launches_per_step(self) -> int:
        n = len(self.cfg.activations())
        for p in self.cfg.projections:
            n += 1 + (1 if p.chained else 0)
            if self.lora:
                n += 4 if p.kind == "gateup" else 2   # each LoRA add is two GEMM launches
                if p.kind == "gateup":
                    n += 1                             # unfused SwiGLU
        return n

    def step(self, acts: Dict[str, torch.Tensor], events=None) -> Dict[str, torch.Tensor]:
        """acts: activation name -> bf16 [M][K].  Returns the output buffers.

        events: optional dict; when given, CUDA events are recorded on the
        current stream around every launch, under keys ("quant", name) and
        ("gemm", name), as (start, end) pairs appended to lists."""
        ev = _Rec(events)
        lin = fp8_linear if self.fp8 else w8a8_linear
        gu = fp8_gateup_swiglu if self.fp8 else w8a8_gateup_swiglu
        for name, _ in self.cfg.activations():
            qx, sx = self.q[name]
            with ev("quant", name):
                quant_act(acts[name], self.mode, q=qx, scale=sx)
        prev_h = None
        for p in self.cfg.projections:
            qw, sw, b = self.w[p.name]
            if p.chained:
                qx, sx = self.q[p.act]
                with ev("quant", p.act):
                    quant_act(prev_h, self.mode, q=qx, scale=sx)
            else:
                qx, sx = self.q[p.act]
            y = self.out[p.name]
            if p.kind == "gateup":
                if self.lora:
                    packed = self.out[p.name + "/packed"]
                    with ev("gemm", p.name):
                        lin(qx, sx, qw, sw, b, y=packed)
                    x = acts[p.act]
                    with ev("lora", p.name):
                        A, B = self.lora[p.name + "/gate"]
                        lora_add(x, A, B, packed[:, :p.N], t_scratch=self._t(A))
                        A, B = self.lora[p.name + "/up"]
                        lora_add(x, A, B, packed[:, p.N:], t_scratch=self._t(A))
                    with ev("swiglu", p.name):
                        swiglu_bf16(packed, h=y)
                else:
                    with ev("gemm", p.name):
                        gu(qx, sx, qw, sw, b, h=y)
                prev_h = y
            else:
                with ev("gemm", p.name):
                    lin(qx, sx, qw, sw, b, y=y)
                if self.lora and p.name in self.lora:
                    A, B = self.lora[p.name]
                    with ev("lora", p.name):
                        lora_add(acts[p.act] if not p.chained else prev_h, A, B, y,
                                 t_scratch=self._t(A))
        return self.out

    def _t(self, A):
        return self.t[lora_pad(A.shape[0])]


class _Rec:
    """Context manager factory recording start/end CUDA events per launch."""

    def __init__(self, events):
        self.events = events

    def __call__(self, kind, name):
        return _Span(self.events, (kind, name))


class _Span:
    def __init__(self, events, key):
        self.events, self.key = events, key

    def __enter__(self):
        if self.events is not None:
            self.s = torch.cuda.Event(enable_timing=True)
            self.s.record()
        return self

    def __exit__(self, *exc):
        if self.events is not None:
            e = torch.cuda.Event(enable_timing=True)
            e.record()
            self.events.setdefault(self.key, []).append((self.s, e))
        return False
