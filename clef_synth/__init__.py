"""Seeded synthetic inputs for the W8A8 projection path.

This module is shared by the CPU oracle tests, the GPU parity tests and the
benchmark, so that both sides of every comparison see the same bytes.  It holds
none of the method's arithmetic (no rotation, no quantisation, no GEMM): only a
counter-based pseudo-random generator, normal deviates and their rounding to
bf16 storage.

Generator (stated so that it can be re-implemented anywhere):

* SplitMix64 (Steele, Lea and Flood, "Fast splittable pseudorandom number
  generators", OOPSLA 2014): the i-th output (i = 1, 2, ...) of stream seed
  ``s`` is ``mix(s + i * 0x9E3779B97F4A7C15)`` with the published mixing
  constants, all arithmetic modulo 2**64.
* One sub-stream per tensor: its seed is the SplitMix64 mix of
  ``seed XOR fnv1a64(name)``.
* Uniforms: the top 53 bits of an output scaled by 2**-53; ``u1`` is shifted to
  (0, 1] so that its logarithm is finite.
* Normals: Box-Muller in fp64, ``sqrt(-2 ln u1) * cos(2 pi u2)``, one normal
  per pair of outputs.
* Storage: the fp64 value (already multiplied by its standard deviation and,
  for outlier channels, by the outlier factor) is rounded to fp32 and then to
  bf16, both round-to-nearest-even; tensors are returned as ``uint16`` arrays
  holding bf16 bit patterns.
"""
from __future__ import annotations

import os
import threading
from concurrent.futures import ThreadPoolExecutor

import numpy as np

from .configs import CONFIGS, WORKLOADS, Config, Projection, workload  # noqa: F401

_GOLDEN = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
_CHUNK = 1 << 22  # normals generated per numpy pass (bounds temporary memory)


def _mix(z: np.ndarray) -> np.ndarray:
    z = (z ^ (z >> np.uint64(30))) * _M1
    z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


def _fnv1a64(name: str) -> int:
    h = 0xCBF29CE484222325
    for b in name.encode("utf-8"):
        h ^= b
        h = (h * 0x100000001B3) & 0xFFFFFFFFFFFFFFFF
    return h


def stream_seed(seed: int, name: str) -> int:
    """Seed of the sub-stream that generates the tensor called ``name``."""
    z = np.array([(seed ^ _fnv1a64(name)) & 0xFFFFFFFFFFFFFFFF], dtype=np.uint64)
    return int(_mix(z)[0])


def splitmix64(seed: int, start: int, n: int) -> np.ndarray:
    """Outputs ``start+1 .. start+n`` of the SplitMix64 stream with this seed."""
    with np.errstate(over="ignore"):
        i = np.arange(start + 1, start + n + 1, dtype=np.uint64)
        z = np.uint64(seed) + i * _GOLDEN
        return _mix(z)


def normals(seed: int, name: str, n: int, start: int = 0) -> np.ndarray:
    """``n`` standard normal deviates (fp64) of the named sub-stream, from index ``start``."""
    s = stream_seed(seed, name)
    z = splitmix64(s, 2 * start, 2 * n)
    scale = 2.0 ** -53
    u1 = ((z[0::2] >> np.uint64(11)).astype(np.float64) + 1.0) * scale
    u2 = (z[1::2] >> np.uint64(11)).astype(np.float64) * scale
    return np.sqrt(-2.0 * np.log(u1)) * np.cos(2.0 * np.pi * u2)


_tls = threading.local()
_BASE = None


def _normals_ws(sseed: np.uint64, start: int, n: int) -> np.ndarray:
    """Same values as ``normals`` for an already-derived stream seed, computed
    in place in a per-thread workspace (fresh pages are slow to fault in)."""
    global _BASE
    if _BASE is None:
        _BASE = np.arange(2 * _CHUNK, dtype=np.uint64)
    ws = getattr(_tls, "ws", None)
    if ws is None:
        ws = _tls.ws = (np.empty(2 * _CHUNK, np.uint64), np.empty(2 * _CHUNK, np.uint64),
                        np.empty(_CHUNK, np.float64), np.empty(_CHUNK, np.float64))
    z, t, u1, u2 = ws
    z, t, u1, u2 = z[:2 * n], t[:2 * n], u1[:n], u2[:n]
    with np.errstate(over="ignore"):
        np.add(_BASE[:2 * n], np.uint64(2 * start + 1), out=z)      # counter i
        np.multiply(z, _GOLDEN, out=z)
        np.add(z, sseed, out=z)
        for sh, mul in ((30, _M1), (27, _M2)):
            np.right_shift(z, np.uint64(sh), out=t)
            np.bitwise_xor(z, t, out=z)
            np.multiply(z, mul, out=z)
        np.right_shift(z, np.uint64(31), out=t)
        np.bitwise_xor(z, t, out=z)
        np.right_shift(z, np.uint64(11), out=z)
    u1[:] = z[0::2]
    u2[:] = z[1::2]
    u1 += 1.0
    u1 *= 2.0 ** -53
    u2 *= 2.0 ** -53
    np.log(u1, out=u1)
    u1 *= -2.0
    np.sqrt(u1, out=u1)
    u2 *= 2.0 * np.pi
    np.cos(u2, out=u2)
    return u1 * u2


def f64_to_bf16_bits(v: np.ndarray) -> np.ndarray:
    """Round fp64 values to bf16 storage (via fp32, both steps nearest-even)."""
    f = np.ascontiguousarray(v, dtype=np.float32).view(np.uint32)
    lsb = (f >> np.uint32(16)) & np.uint32(1)
    with np.errstate(over="ignore"):
        r = (f + np.uint32(0x7FFF) + lsb) >> np.uint32(16)
    return r.astype(np.uint16)


def bf16_bits_to_f64(b: np.ndarray) -> np.ndarray:
    """Exact value of bf16 bit patterns, as fp64."""
    return (b.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


def outlier_channels(seed: int, name: str, K: int, count: int = 8) -> np.ndarray:
    """``count`` distinct channel indices in [0, K), by a partial Fisher-Yates shuffle."""
    count = min(count, K)
    perm = np.arange(K, dtype=np.int64)
    r = splitmix64(stream_seed(seed, name + "/outliers"), 0, count)
    for i in range(count):
        j = i + int(r[i] % np.uint64(K - i))
        perm[i], perm[j] = perm[j], perm[i]
    return np.sort(perm[:count])


def normal_bf16(seed: int, name: str, shape, std: float = 1.0,
                outliers: int = 0, outlier_scale: float = 20.0) -> np.ndarray:
    """A bf16 tensor (uint16 bits) of N(0, std^2) entries, row-major ``shape``.

    With ``outliers > 0`` the last axis gets that many distinct outlier
    channels whose entries are multiplied by ``outlier_scale`` before rounding.
    """
    shape = tuple(int(d) for d in shape)
    n = int(np.prod(shape)) if shape else 1
    out = np.empty(n, dtype=np.uint16)
    cols = None
    if outliers:
        K = shape[-1]
        mult = np.ones(K, dtype=np.float64)
        mult[outlier_channels(seed, name, K, outliers)] = outlier_scale
        cols = mult
    sseed = np.uint64(stream_seed(seed, name))

    def fill(a):
        b = min(n, a + _CHUNK)
        v = _normals_ws(sseed, a, b - a)
        v *= std
        if cols is not None:
            v *= cols[np.arange(a, b, dtype=np.int64) % shape[-1]]
        out[a:b] = f64_to_bf16_bits(v)

    starts = range(0, n, _CHUNK)
    if n > _CHUNK:
        with ThreadPoolExecutor(max_workers=min(16, os.cpu_count() or 1)) as ex:
            list(ex.map(fill, starts))
    else:
        for a in starts:
            fill(a)
    return out.reshape(shape)


def activation(seed: int, name: str, M: int, K: int) -> np.ndarray:
    """Activation rows: N(0,1) with 8 outlier channels scaled by 20."""
    return normal_bf16(seed, name, (M, K), 1.0, outliers=8, outlier_scale=20.0)


def weight(seed: int, name: str, N: int, K: int) -> np.ndarray:
    """Projection weight ``[N][K]`` (output channel major): N(0, 0.02^2)."""
    return normal_bf16(seed, name, (N, K), 0.02)


def bias(seed: int, name: str, N: int) -> np.ndarray:
    """Projection bias ``[N]``: N(0, 0.01^2)."""
    return normal_bf16(seed, name, (N,), 0.01)


def lora_pair(seed: int, name: str, r: int, K: int, N: int):
    """LoRA factors A ``[r][K]`` and B ``[N][r]``, entries N(0, 0.01^2)."""
    return (normal_bf16(seed, name + "/A", (r, K), 0.01),
            normal_bf16(seed, name + "/B", (N, r), 0.01))


def layer_inputs(cfg: Config, seed: int = 0, rows: slice | None = None):
    """Seeded inputs of one workload: activations, weights (+bias) and LoRA pairs.

    Returns (acts, weights, lora) as numpy bf16-bit arrays:
    acts[name] = [M][K] (chained inputs are produced by the path itself and are
    absent); weights[proj] = (W [rows][K], bias [rows]) with gate/up packed gate
    rows first; lora[proj] = (A [r][K], B [N][r]) and, for gate/up,
    lora[proj + "/gate"], lora[proj + "/up"].  Every tensor has its own named
    sub-stream, so any subset can be regenerated alone.
    """
    acts = {}
    for name, K in cfg.activations():
        acts[name] = activation(seed, f"{cfg.name}/act/{name}", cfg.M, K)
    weights, lora = {}, {}
    for p in cfg.projections:
        if p.kind == "gateup":
            W = np.concatenate([weight(seed, f"{cfg.name}/w/{p.name}/gate", p.N, p.K),
                                weight(seed, f"{cfg.name}/w/{p.name}/up", p.N, p.K)])
            b = np.concatenate([bias(seed, f"{cfg.name}/b/{p.name}/gate", p.N),
                                bias(seed, f"{cfg.name}/b/{p.name}/up", p.N)])
        else:
            W = weight(seed, f"{cfg.name}/w/{p.name}", p.N, p.K)
            b = bias(seed, f"{cfg.name}/b/{p.name}", p.N)
        weights[p.name] = (W, b)
        if cfg.lora_rank:
            r = cfg.lora_rank
            if p.kind == "gateup":
                lora[p.name + "/gate"] = lora_pair(seed, f"{cfg.name}/lora/{p.name}/gate", r, p.K, p.N)
                lora[p.name + "/up"] = lora_pair(seed, f"{cfg.name}/lora/{p.name}/up", r, p.K, p.N)
            else:
                lora[p.name] = lora_pair(seed, f"{cfg.name}/lora/{p.name}", r, p.K, p.N)
    return acts, weights, lora
