"""Seeded synthetic inputs for the MoE expert layer.

This module only draws numbers. It holds none of the layer's arithmetic (no routing,
no layout, no expert math), so both the CUDA path and the CPU oracle can take their
inputs from it without sharing any computation.

Recipe (the workloads of the tile-level signaling MoE page, "The pith" and
"Core claim": an MoE layer whose tokens come from R source partitions):

* router logits: float32, N(0, 1) per entry; the skewed workload adds a per-expert
  bias b_e = 2 * ln(1 / (e + 1) ** 1.2) (a Zipf-like load) in float32;
* token activations x: N(0, 1) drawn in float32, rounded to bfloat16
  (round-to-nearest-even);
* expert weights W1, W3 of shape [E, ffn, d] and W2 of shape [E, d, ffn]:
  N(0, 1/d) drawn in float32, rounded to bfloat16.

Every tensor is split into fixed chunks of 2**20 elements; chunk i of tensor ``tag``
is drawn from ``numpy.random.default_rng(SeedSequence([seed, tag, i]))``. The result
therefore does not depend on how many threads draw it, and any slice of a large
tensor can be regenerated on its own.
"""
from __future__ import annotations

import dataclasses
import math
import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import torch

CHUNK = 1 << 20

# tensor tags of the chunked generator
TAG_LOGITS, TAG_X, TAG_W1, TAG_W3, TAG_W2 = 1, 2, 3, 4, 5


@dataclasses.dataclass(frozen=True)
class Workload:
    """Shape of one MoE layer workload.

    T tokens of width d, E experts of hidden width ffn, top-k routing, R owner
    partitions of the tokens (contiguous, T/R each), GEMM tile height tile_M.
    """

    name: str
    T: int
    d: int
    ffn: int
    E: int
    topk: int
    R: int
    tile_M: int
    skew: bool = False

    def replace(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


# The four layer shapes that are measured and parity-tested.
WORKLOADS = {
    "tiny": Workload("tiny", T=256, d=128, ffn=256, E=4, topk=2, R=2, tile_M=64),
    "mixtral": Workload("mixtral", T=4096, d=4096, ffn=14336, E=8, topk=2, R=4, tile_M=128),
    "skew": Workload("skew", T=8192, d=2048, ffn=5632, E=16, topk=2, R=8, tile_M=128, skew=True),
    "fine": Workload("fine", T=16384, d=2048, ffn=1408, E=64, topk=6, R=8, tile_M=128),
}


def _threads() -> int:
    return max(1, min(16, os.cpu_count() or 1))


def normal_f32(n: int, seed: int, tag: int, std: float = 1.0, start: int = 0) -> np.ndarray:
    """Elements [start, start+n) of the chunked N(0, std^2) float32 stream (seed, tag)."""
    out = np.empty(n, np.float32)
    if n == 0:
        return out
    c0, c1 = start // CHUNK, (start + n - 1) // CHUNK

    def fill(c: int) -> None:
        rng = np.random.default_rng(np.random.SeedSequence([seed, tag, c]))
        lo, hi = c * CHUNK, (c + 1) * CHUNK
        a, b = max(lo, start), min(hi, start + n)
        if a == lo and b == hi:
            rng.standard_normal(out=out[a - start:b - start], dtype=np.float32)
        else:
            full = rng.standard_normal(CHUNK, dtype=np.float32)
            out[a - start:b - start] = full[a - lo:b - lo]

    chunks = range(c0, c1 + 1)
    if len(chunks) == 1:
        fill(c0)
    else:
        with ThreadPoolExecutor(_threads()) as ex:
            list(ex.map(fill, chunks))
    if std != 1.0:
        out *= np.float32(std)
    return out


def to_bf16(a: np.ndarray) -> torch.Tensor:
    """float32 array -> bfloat16 CPU tensor, round-to-nearest-even (torch's conversion)."""
    return torch.from_numpy(np.ascontiguousarray(a, np.float32)).to(torch.bfloat16)


def expert_bias(E: int) -> np.ndarray:
    """Zipf-like per-expert router bias b_e = 2 ln(1/(e+1)^1.2), float32."""
    e = np.arange(E, dtype=np.float64)
    return (2.0 * np.log(1.0 / (e + 1.0) ** 1.2)).astype(np.float32)


def make_logits(w: Workload, seed: int) -> np.ndarray:
    """Router logits, float32 [T, E]."""
    l = normal_f32(w.T * w.E, seed, TAG_LOGITS).reshape(w.T, w.E)
    if w.skew:
        l = l + expert_bias(w.E)[None, :]
    return l


def make_x(w: Workload, seed: int) -> torch.Tensor:
    """Token activations, bfloat16 [T, d] (CPU)."""
    return to_bf16(normal_f32(w.T * w.d, seed, TAG_X)).reshape(w.T, w.d)


def make_weight(w: Workload, seed: int, which: str, experts: range | None = None) -> torch.Tensor:
    """One expert weight tensor as bfloat16 on the CPU.

    which: "W1" or "W3" -> [E, ffn, d]; "W2" -> [E, d, ffn]. ``experts`` selects a
    subset of experts (the generator regenerates only their chunks).
    """
    tag = {"W1": TAG_W1, "W3": TAG_W3, "W2": TAG_W2}[which]
    per = w.ffn * w.d
    shape = (w.ffn, w.d) if which != "W2" else (w.d, w.ffn)
    ex = range(w.E) if experts is None else experts
    std = 1.0 / math.sqrt(w.d)
    parts = [to_bf16(normal_f32(per, seed, tag, std, start=e * per)).reshape(shape) for e in ex]
    return torch.stack(parts) if parts else torch.empty((0,) + shape, dtype=torch.bfloat16)


def make_weight_into(w: Workload, seed: int, which: str, dst: torch.Tensor) -> None:
    """Fill ``dst`` (any device, [E, ...] bf16) expert by expert, bounding host memory."""
    for e in range(w.E):
        dst[e].copy_(make_weight(w, seed, which, range(e, e + 1))[0])


def make_all(w: Workload, seed: int) -> dict:
    """All inputs of one layer on the CPU: logits (numpy f32) and bf16 torch tensors."""
    return {
        "logits": make_logits(w, seed),
        "x": make_x(w, seed),
        "W1": make_weight(w, seed, "W1"),
        "W3": make_weight(w, seed, "W3"),
        "W2": make_weight(w, seed, "W2"),
    }


def bf16_to_f64(t: torch.Tensor) -> np.ndarray:
    """Exact widening of a bfloat16 tensor to a float64 numpy array."""
    return t.detach().to("cpu").to(torch.float64).numpy()
