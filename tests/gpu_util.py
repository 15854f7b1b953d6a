"""Helpers shared by the GPU parity tests: moving seeded inputs between numpy
(bf16 as uint16 bits) and CUDA tensors, bf16 ulp comparisons, and running
oracle functions over row slices on all host cores (ctypes releases the GIL,
so threads run the single-threaded C oracle in parallel)."""
from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import torch

import clef_synth as S

THREADS = max(1, min(32, os.cpu_count() or 1))


def bf16_dev(u16: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(u16).view(np.int16)).view(torch.bfloat16).cuda()


def bf16_host(t: torch.Tensor) -> np.ndarray:
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


def dev(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def host(t: torch.Tensor) -> np.ndarray:
    return t.detach().contiguous().cpu().numpy()


def bf16_ulp(v):
    a = np.maximum(np.abs(np.asarray(v, np.float64)), 2.0 ** -126)
    return 2.0 ** (np.floor(np.log2(a)) - 7)


def ulp_diff(got_u16: np.ndarray, ref_u16: np.ndarray) -> np.ndarray:
    """|got - ref| in units of the bf16 ulp at ref."""
    g, r = S.bf16_bits_to_f64(got_u16), S.bf16_bits_to_f64(ref_u16)
    return np.abs(g - r) / bf16_ulp(r)


def assert_bf16_within(got_u16, ref_u16, ulps: float = 1.0, what: str = ""):
    d = ulp_diff(got_u16, ref_u16)
    bad = d > ulps
    if bad.any():
        idx = np.argwhere(bad)[:5].tolist()
        raise AssertionError(f"{what}: {int(bad.sum())} of {d.size} outside {ulps} ulp, "
                             f"worst {d.max():.2f} ulp, first at {idx}")


def par_rows(fn, M: int, chunk: int | None = None):
    """Concatenate fn(a, b) over row ranges [a, b) covering [0, M), in threads."""
    if M == 0:
        return fn(0, 0)
    chunk = chunk or max(1, -(-M // THREADS))
    ranges = [(a, min(M, a + chunk)) for a in range(0, M, chunk)]
    with ThreadPoolExecutor(max_workers=THREADS) as ex:
        parts = list(ex.map(lambda ab: fn(*ab), ranges))
    if isinstance(parts[0], tuple):
        return tuple(np.concatenate([p[i] for p in parts]) for i in range(len(parts[0])))
    return np.concatenate(parts)
