"""One decoder layer's quantized projections, run through the C ABI.

``QuantizedLayer`` quantizes the bf16 weights once at set-up with the same
quantizer the activations use (INT8: block-128 rotation and per-output-channel
scales; FP8: per-channel e4m3 from the weights alone, as the "clef-flash-FP8"
model card's Quantization table describes), packs gate and up side by side
(gate rows first, as the "Loading CLEF INT8" usage notes pack them at load),
and preallocates every activation-code, scale, scratch and output buffer so
that a ``step`` launches kernels only.

Consecutive plain projections that read the same activation (q, k and v read
the same hidden state) are packed the same way: their weight rows, scales
and biases are stacked at set-up and one GEMM call writes all of their
outputs into one [M][N_q + N_k + N_v] buffer, of which each projection's
output is a column slice.  Every output element is the same function of the
same row and column as in separate calls (per-row scales, per-output-channel
weight scales, no split of K), so packing changes no bit; it only gives the
small k and v projections the tile count of one wide GEMM.

A step runs, per distinct activation tensor, one quantizer call, then per
projection one GEMM call (gate/up with the fused SwiGLU epilogue).  With
runtime LoRA pairs, every adapted projection adds ``bf16(x A^T) B^T`` after
its GEMM; gate/up is then run as a packed linear (bf16 gate and up), and one
call adds the gate and up adapters to their halves and forms h (the same
rounded operations as two LoRA adds followed by the unfused SwiGLU).  The
adapters of a packed group share their input, so their A factors are stacked
at set-up (each padded to 64 rows) and one shrink call computes every
adapter's t from one pass over x; each adapter's expand call then reads its
own column block of t (the same bytes as a separate LoRA add per adapter).
"""
from __future__ import annotations

from types import SimpleNamespace
from typing import Dict, Optional, Tuple

import torch

from . import (bind_workspace, fp8_gateup_swiglu, fp8_linear, gemm_workspace_bytes, lora_add,
               lora_expand_add, lora_gateup_swiglu, lora_pad, lora_shrink, poll_status, quant_act,
               w8a8_gateup_swiglu, w8a8_gateup_swiglu_lora, w8a8_linear, w8a8_linear_lora)

TIMEOUT = 4   # CLEF_ERR_TIMEOUT


class QuantizedLayer:
    def __init__(self, cfg, weights: Dict[str, Tuple[torch.Tensor, Optional[torch.Tensor]]],
                 lora: Optional[Dict[str, Tuple[torch.Tensor, torch.Tensor]]] = None,
                 device="cuda", pack_shared_input: bool = True, fuse_lora: bool = True):
        """weights: projection name -> (W bf16 [rows][K], bias bf16 [rows] or None);
        lora: name (or name + "/gate", name + "/up" for gate/up) -> (A, B);
        pack_shared_input: run consecutive plain projections of one activation
        as one packed GEMM;
        fuse_lora (INT8): add each adapted launch unit's LoRA inside its GEMM
        (one x A^T launch, then the GEMM with the expand fused; for gate/up
        before the SwiGLU) instead of adapter launches over the GEMM's
        output; the bytes are the same."""
        self.cfg = cfg
        self.M = cfg.M
        self.fp8 = cfg.scheme == "fp8"
        self.mode = "fp8" if self.fp8 else "int8_h128"
        self.lora = lora or {}
        M = self.M
        self.groups = _groups(cfg.projections, weights) if pack_shared_input else \
            [[p] for p in cfg.projections]
        # quantized weights per launch unit; self.w[name] are row views of them
        self.w = {}
        self.unit_w = []
        for g in self.groups:
            if len(g) == 1:
                W, b = weights[g[0].name]
            else:
                W = torch.cat([weights[p.name][0] for p in g], dim=0)
                bs = [weights[p.name][1] for p in g]
                b = None if bs[0] is None else torch.cat(bs, dim=0)
            qw, sw = quant_act(W, self.mode)
            self.unit_w.append((qw, sw, b))
            r0 = 0
            for p in g:
                r1 = r0 + p.weight_rows
                self.w[p.name] = (qw[r0:r1], sw[r0:r1], None if b is None else b[r0:r1])
                r0 = r1
        torch.cuda.synchronize()
        # a stream-K workspace, bound to whichever stream runs a step (tiles of
        # a GEMM whose last wave would be mostly idle are split across SMs: the
        # INT8 GEMMs' exact int32 pieces, the FP8 linear's fixed K halves; the
        # outputs are the same bytes)
        self.ws = torch.zeros(gemm_workspace_bytes(), dtype=torch.uint8, device=device)
        self._ws_stream = None   # the stream the workspace was last bound to
        # fused LoRA (INT8): per adapted launch unit, its stacked A factors, its
        # t, its stacked B factor(s) and the column segments of its adapters
        self.fused = {}
        if fuse_lora and not self.fp8 and self.lora:
            for gi, g in enumerate(self.groups):
                f = _fused_unit(g, self.lora, M, device)
                if f is not None:
                    self.fused[gi] = f
        fused_names = {p.name for gi in self.fused for p in self.groups[gi]}
        code = torch.uint8 if self.fp8 else torch.int8
        self.q = {}
        for name, K in cfg.activations():
            self.q[name] = (torch.empty((M, K), dtype=code, device=device),
                            torch.empty((M,), dtype=torch.float32, device=device))
        self.out = {}
        self.unit_out = []
        for g in self.groups:
            if len(g) > 1:
                packed = torch.empty((M, sum(p.N for p in g)), dtype=torch.bfloat16, device=device)
                self.unit_out.append(packed)
                c0 = 0
                for p in g:
                    self.out[p.name] = packed[:, c0:c0 + p.N]
                    c0 += p.N
            else:
                self.unit_out.append(None)
        for p in cfg.projections:
            if p.name in self.out:
                continue
            if p.kind == "gateup":
                self.out[p.name] = torch.empty((M, p.N), dtype=torch.bfloat16, device=device)
                if self.lora and p.name not in fused_names:
                    self.out[p.name + "/packed"] = torch.empty((M, 2 * p.N), dtype=torch.bfloat16,
                                                               device=device)
            else:
                self.out[p.name] = torch.empty((M, p.N), dtype=torch.bfloat16, device=device)
            if p.chained:
                self.q[p.act] = (torch.empty((M, p.K), dtype=code, device=device),
                                 torch.empty((M,), dtype=torch.float32, device=device))
        # LoRA scratch: per packed group with adapters, the stacked A factors
        # and a [M][sum r_pad] t whose column blocks belong to its adapters;
        # one dense [M][r_pad] (or [M][2 r_pad] for the gate/up pair) per width
        # for the others
        self.t = {}
        self.lora_groups = {}   # group index -> (stacked A, t, [(name, col0, r_pad)])
        for gi, g in enumerate(self.groups):
            members = [p for p in g if p.name in self.lora] if len(g) > 1 and gi not in self.fused else []
            if not members:
                continue
            K = g[0].K
            pads = [lora_pad(self.lora[p.name][0].shape[0]) for p in members]
            A_cat = torch.zeros((sum(pads), K), dtype=torch.bfloat16, device=device)
            blocks, c0 = [], 0
            for p, r_pad in zip(members, pads):
                A = self.lora[p.name][0]
                A_cat[c0:c0 + A.shape[0]] = A
                blocks.append((p.name, c0, r_pad))
                c0 += r_pad
            t = torch.empty((M, c0), dtype=torch.bfloat16, device=device)
            self.lora_groups[gi] = (A_cat, t, blocks)
        grouped = {name for _, _, blocks in self.lora_groups.values() for name, _, _ in blocks}
        for key, (A, _) in self.lora.items():
            if key in grouped or key.split("/")[0] in fused_names:
                continue
            width = lora_pad(A.shape[0]) * (2 if key.endswith("/gate") or key.endswith("/up") else 1)
            if width not in self.t:
                self.t[width] = torch.empty((M, width), dtype=torch.bfloat16, device=device)

    def units(self):
        """The GEMM launches of a step: (event name, weight rows, K, 2*M*rows*K,
        the flops of the LoRA expand fused into the launch: 2*M*N*r per adapter)."""
        out = []
        for gi, g in enumerate(self.groups):
            rows = sum(p.weight_rows for p in g)
            fused = 0
            if gi in self.fused:
                for p in g:
                    for key in ((p.name + "/gate", p.name + "/up") if p.kind == "gateup" else (p.name,)):
                        if key in self.lora:
                            N, r = self.lora[key][1].shape
                            fused += 2 * self.M * N * r
            out.append((_unit_name(g), rows, g[0].K, 2 * self.M * rows * g[0].K, fused))
        return out

    def lora_work(self) -> Tuple[int, int]:
        """Per step, the LoRA launches' (flops, minimum HBM bytes): 2 M r (K + N)
        flops per adapter; x read once per shrink launch, t written and read
        back, y read and written (gate/up: both base halves read, h written)."""
        M, fl, by = self.M, 0, 0
        for gi, g in enumerate(self.groups):
            if gi in self.fused:
                # fused: the LoRA launch is x A^T alone (x read, t written); the
                # expand's flops belong to the GEMM (units())
                f = self.fused[gi]
                by += M * g[0].K * 2 + M * f.t.shape[1] * 2
                for p in g:
                    for key in ((p.name + "/gate", p.name + "/up") if p.kind == "gateup" else (p.name,)):
                        if key in self.lora:
                            fl += 2 * M * self.lora[key][0].shape[0] * p.K
                continue
            if gi in self.lora_groups:
                _, t, blocks = self.lora_groups[gi]
                by += M * g[0].K * 2 + 2 * M * t.shape[1] * 2
                for name, _, _ in blocks:
                    N, r = self.lora[name][1].shape
                    fl += 2 * M * r * (g[0].K + N)
                    by += 2 * M * N * 2
                continue
            for p in g:
                if p.kind == "gateup" and p.name + "/gate" in self.lora:
                    for half in ("/gate", "/up"):
                        A, B = self.lora[p.name + half]
                        fl += 2 * M * A.shape[0] * (p.K + B.shape[0])
                    r_pad = lora_pad(self.lora[p.name + "/gate"][0].shape[0])
                    by += M * p.K * 2 + 2 * M * 2 * r_pad * 2 + M * 2 * p.N * 2 + M * p.N * 2
                elif p.name in self.lora:
                    A, B = self.lora[p.name]
                    fl += 2 * M * A.shape[0] * (p.K + B.shape[0])
                    by += M * p.K * 2 + 2 * M * lora_pad(A.shape[0]) * 2 + 2 * M * B.shape[0] * 2
        return fl, by

    def launches_per_step(self) -> int:
        n = len(self.cfg.activations()) + len(self.groups)
        for p in self.cfg.projections:
            n += 1 if p.chained else 0
        if self.lora:
            for gi, g in enumerate(self.groups):
                if gi in self.fused:            # x A^T, then the GEMM with the expand fused
                    n += 1
                elif gi in self.lora_groups:    # one shared x A^T, one expand per adapter
                    n += 1 + len(self.lora_groups[gi][2])
                elif g[0].kind == "gateup":     # stacked x A^T, one fused add + SwiGLU
                    n += 2
                else:
                    n += sum(2 for p in g if p.name in self.lora)
        return n

    def step(self, acts: Dict[str, torch.Tensor], events=None,
             final_wait: Optional[torch.cuda.Event] = None) -> Dict[str, torch.Tensor]:
        """acts: activation name -> bf16 [M][K].  Returns the output buffers.

        events: optional dict; when given, CUDA events are recorded on the
        current stream around every launch, under keys ("quant", name),
        ("gemm", name) and ("lora", name) (a packed group's shared x A^T under
        ("lora", "q+k+v:xA")), as (start, end) pairs appended to lists.
        final_wait: optional CUDA event the current stream waits for before the
        step's last projection writes its output (e.g. the read-back of the
        previous step's output on another stream)."""
        ev = _Rec(events)
        if self.ws is not None:
            # bind once per stream (the binding is host bookkeeping, but a
            # Python call per step would delay the step's first launch)
            s = torch.cuda.current_stream()
            if self._ws_stream != s.cuda_stream:
                bind_workspace(self.ws, s)
                self._ws_stream = s.cuda_stream
        lin = fp8_linear if self.fp8 else w8a8_linear
        gu = fp8_gateup_swiglu if self.fp8 else w8a8_gateup_swiglu
        for name, _ in self.cfg.activations():
            qx, sx = self.q[name]
            with ev("quant", name):
                quant_act(acts[name], self.mode, q=qx, scale=sx)
        prev_h = None
        last = len(self.groups) - 1
        for gi, g in enumerate(self.groups):
            if gi == last and final_wait is not None:
                torch.cuda.current_stream().wait_event(final_wait)
            if gi in self.fused:
                prev_h = self._step_fused(gi, g, acts, prev_h, ev)
                continue
            if len(g) > 1:
                qw, sw, b = self.unit_w[gi]
                qx, sx = self.q[g[0].act]
                with ev("gemm", _unit_name(g)):
                    lin(qx, sx, qw, sw, b, y=self.unit_out[gi])
                if gi in self.lora_groups:
                    A_cat, t, blocks = self.lora_groups[gi]
                    with ev("lora", _unit_name(g) + ":xA"):
                        lora_shrink(acts[g[0].act], A_cat, t=t)
                    for name, c0, r_pad in blocks:
                        with ev("lora", name):
                            lora_expand_add(t[:, c0:c0 + r_pad], self.lora[name][1], self.out[name])
                continue
            p = g[0]
            qw, sw, b = self.unit_w[gi]
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
                    Ag, Bg = self.lora[p.name + "/gate"]
                    Au, Bu = self.lora[p.name + "/up"]
                    with ev("lora", p.name):
                        lora_gateup_swiglu(acts[p.act], Ag, Bg, Au, Bu, packed, h=y,
                                           t_scratch=self.t[2 * lora_pad(Ag.shape[0])])
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

    def _step_fused(self, gi, g, acts, prev_h, ev):
        """One launch unit with its LoRA fused: x A^T for all of the unit's
        adapters in one launch, then the INT8 GEMM whose tiles add t B^T to
        their rounded base values (gate/up: before the SwiGLU)."""
        f = self.fused[gi]
        qw, sw, b = self.unit_w[gi]
        p = g[0]
        name = _unit_name(g)
        x = prev_h if p.chained else acts[p.act]
        if p.chained:
            qx, sx = self.q[p.act]
            with ev("quant", p.act):
                quant_act(prev_h, self.mode, q=qx, scale=sx)
        else:
            qx, sx = self.q[p.act]
        with ev("lora", name + ":xA"):
            lora_shrink(x, f.A, t=f.t)
        if p.kind == "gateup":
            with ev("gemm", name):
                w8a8_gateup_swiglu_lora(qx, sx, qw, sw, b, f.t, f.B, f.B_up, h=self.out[p.name])
            return self.out[p.name]
        y = self.unit_out[gi] if len(g) > 1 else self.out[p.name]
        with ev("gemm", name):
            w8a8_linear_lora(qx, sx, qw, sw, b, f.t, f.B, y=y, segments=f.segments)
        return prev_h

    def poll_status(self) -> int:
        """Synchronise, then return (and clear) the library's device status
        word.  After a device-side time-out the stream-K workspace may hold
        arrival counts of pieces that never arrived (a CTA pair that gave up
        partway through a split tile), which would make a later launch finish
        that tile early or never; so on CLEF_ERR_TIMEOUT the workspace is
        refilled with zeros here, before any further step (a captured graph
        keeps the same buffer, so its replays see the refill too)."""
        st = poll_status()
        if st == TIMEOUT and self.ws is not None:
            self.ws.zero_()
            torch.cuda.synchronize(self.ws.device)
        return st

    def capture(self, acts: Dict[str, torch.Tensor]) -> "torch.cuda.CUDAGraph":
        """Record one step on ``acts`` into a CUDA graph (after a warm-up step
        on a side stream, which performs the library's one-time per-device and
        per-kernel set-up outside the capture).  ``replay()`` then reruns the
        step's launches on the same input and output buffers with one launch
        of the graph; refill the input tensors in place to step on new data."""
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            self.step(acts)
        torch.cuda.current_stream().wait_stream(side)
        torch.cuda.synchronize()
        self._unbind()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            self.step(acts)
            # the graph keeps the workspace's address; drop the host binding of
            # the capture stream so no later user of that stream inherits it
            self._unbind()
        self.graph = graph
        return graph

    def _unbind(self):
        if self.ws is not None and self._ws_stream is not None:
            bind_workspace(None, SimpleNamespace(cuda_stream=self._ws_stream))
            self._ws_stream = None

    def replay(self) -> Dict[str, torch.Tensor]:
        self.graph.replay()
        return self.out

    def _t(self, A):
        return self.t[lora_pad(A.shape[0])]


def _fused_unit(g, lora, M, device):
    """The fused-LoRA buffers of one launch unit, or None when it has no
    adapter or its adapters cannot share one fused launch (different ranks,
    more than four adapters, or column segments off the 256-column tiles).

    Linear units: A = the adapters' A factors stacked, each padded with zero
    rows to r_pad; t = [M][sum r_pad]; B = [N_unit][r] with each adapter's B
    rows at its projection's output columns (zero rows for a projection
    without an adapter, which then adds exact zeros); segments map each
    projection's columns to its t block.  Gate/up: A = [A_gate; A_up], t =
    [M][2 r_pad], and the two B factors."""
    if g[0].kind == "gateup":
        p = g[0]
        if p.name + "/gate" not in lora:
            return None
        (Ag, Bg), (Au, Bu) = lora[p.name + "/gate"], lora[p.name + "/up"]
        r = Ag.shape[0]
        if Au.shape[0] != r or Bg.shape[1] != r or Bu.shape[1] != r:
            return None
        rp = lora_pad(r)
        A = torch.zeros((2 * rp, p.K), dtype=torch.bfloat16, device=device)
        A[:r] = Ag
        A[rp:rp + r] = Au
        t = torch.empty((M, 2 * rp), dtype=torch.bfloat16, device=device)
        return SimpleNamespace(A=A, t=t, B=Bg.contiguous(), B_up=Bu.contiguous(), segments=None)
    members = [p for p in g if p.name in lora]
    if not members:
        return None
    ranks = {lora[p.name][0].shape[0] for p in members}
    if len(ranks) != 1 or len(g) > 4:
        return None
    r = ranks.pop()
    rp = lora_pad(r)
    K = g[0].K
    A = torch.zeros((rp * len(members), K), dtype=torch.bfloat16, device=device)
    B = torch.zeros((sum(p.N for p in g), r), dtype=torch.bfloat16, device=device)
    segments, c0, tb = [], 0, 0
    for p in g:
        if p.name in lora:
            Ap, Bp = lora[p.name]
            A[tb:tb + r] = Ap
            B[c0:c0 + p.N] = Bp
            tcol, tb = tb, tb + rp
        else:
            tcol = 0     # its B rows are zeros
        c0 += p.N
        if c0 % 256 != 0 and p is not g[-1]:
            return None
        segments.append((c0, tcol))
    t = torch.empty((M, tb), dtype=torch.bfloat16, device=device)
    return SimpleNamespace(A=A, t=t, B=B, B_up=None, segments=segments)


def _unit_name(group) -> str:
    return "+".join(p.name for p in group)


def _groups(projections, weights):
    """Runs of consecutive plain, unchained projections reading the same
    activation with the same K (and all with or all without bias)."""
    groups = []
    for p in projections:
        g = groups[-1] if groups else None
        if (g is not None and p.kind == "linear" and not p.chained and g[-1].kind == "linear"
                and not g[-1].chained and g[-1].act == p.act and g[-1].K == p.K
                and (weights[g[-1].name][1] is None) == (weights[p.name][1] is None)):
            g.append(p)
        else:
            groups.append([p])
    return groups


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
