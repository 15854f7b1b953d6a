"""Shapes of the five synthetic workloads of the W8A8 projection path.

Each workload is a list of projections of one decoder layer at a token count
``M``.  ``kind`` is ``"linear"`` (one output per weight row) or ``"gateup"``
(gate rows and up rows packed side by side, ``N`` is the width of each half).
``act`` names the activation tensor a projection reads; projections that name
the same activation share it (q, k and v read the same hidden state).
``chained`` marks a ``down`` projection whose input is the SwiGLU output of
the preceding gate/up projection rather than an independent tensor.

The token counts 298, 1,502 and 2,270 are the input lengths of the latency
table on the INT8 ConvRot model card ("Input Tokens" table); 24,032 is sixteen
records of 1,502 tokens, the equal-length batches of its throughput note.
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import List, Optional


@dataclass(frozen=True)
class Projection:
    name: str
    K: int
    N: int
    kind: str = "linear"          # "linear" | "gateup"
    act: str = "x"
    chained: bool = False

    @property
    def weight_rows(self) -> int:
        return 2 * self.N if self.kind == "gateup" else self.N

    def ops(self, M: int) -> int:
        """Algorithmic multiply-add count times two (2*M*rows*K)."""
        return 2 * M * self.weight_rows * self.K


@dataclass(frozen=True)
class Config:
    index: int
    name: str
    M: int
    scheme: str                    # "int8" | "fp8"
    projections: List[Projection] = field(default_factory=list)
    lora_rank: Optional[int] = None

    def activations(self):
        """Distinct (name, K) activation inputs, in first-use order."""
        seen, out = set(), []
        for p in self.projections:
            if p.chained or p.act in seen:
                continue
            seen.add(p.act)
            out.append((p.act, p.K))
        return out

    def gemm_ops(self) -> int:
        return sum(p.ops(self.M) for p in self.projections)

    def lora_flops(self) -> int:
        if not self.lora_rank:
            return 0
        tot = 0
        for p in self.projections:
            n_out = p.weight_rows
            if p.kind == "gateup":
                # one pair per half: gate and up each get A [r][K], B [N][r]
                tot += 2 * (2 * self.M * self.lora_rank * (p.K + p.N))
            else:
                tot += 2 * self.M * self.lora_rank * (p.K + n_out)
        return tot


def _layer27b(M: int) -> List[Projection]:
    return [
        Projection("q", 5120, 6144, act="x_attn"),
        Projection("k", 5120, 1024, act="x_attn"),
        Projection("v", 5120, 1024, act="x_attn"),
        Projection("o", 6144, 5120, act="x_o"),
        Projection("gateup", 5120, 17408, kind="gateup", act="x_mlp"),
        Projection("down", 17408, 5120, act="x_down"),
    ]


def _layer9b() -> List[Projection]:
    return [
        Projection("q", 4096, 4096, act="x_attn"),
        Projection("k", 4096, 1024, act="x_attn"),
        Projection("v", 4096, 1024, act="x_attn"),
        Projection("o", 4096, 4096, act="x_o"),
        Projection("gateup", 4096, 12288, kind="gateup", act="x_mlp"),
        Projection("down", 12288, 4096, act="x_down"),
    ]


CONFIGS = {
    0: Config(0, "int8-linear-m298-2048x2048", 298, "int8",
              [Projection("proj", 2048, 2048, act="x")]),
    1: Config(1, "int8-mlp-27b-m1502", 1502, "int8",
              [Projection("gateup", 5120, 17408, kind="gateup", act="x_mlp"),
               Projection("down", 17408, 5120, act="h", chained=True)]),
    2: Config(2, "int8-layer-27b-m2270", 2270, "int8", _layer27b(2270)),
    3: Config(3, "fp8-layer-9b-m1502", 1502, "fp8", _layer9b()),
    4: Config(4, "int8-layer-27b-m24032-lora256", 24032, "int8", _layer27b(24032),
              lora_rank=256),
}

WORKLOADS = {c.name: c for c in CONFIGS.values()}


def workload(key) -> Config:
    """The workload called ``key`` (its name), or at position ``key`` (0-4)."""
    if isinstance(key, int) or (isinstance(key, str) and key.isdigit()):
        return CONFIGS[int(key)]
    if key not in WORKLOADS:
        raise KeyError(f"unknown workload {key!r}; known: {', '.join(WORKLOADS)}")
    return WORKLOADS[key]
