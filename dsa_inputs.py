"""Seeded synthetic inputs for the DSA layer workloads.

This module only draws random numbers and names the workload shapes.  It
holds none of the layer's arithmetic, so both the CPU oracle and the CUDA
library can be fed from it without sharing any of the method.

Workloads (one DeepSeek Sparse Attention layer, MQA: Hq query heads share one
K/V head; the indexer has Hi heads of width di; pools of 4 tokens):

  tiny_fp32_fwd      L=4096,   Hq=8,  d=64,  Hi=4, di=64,  k=64,  fp32, forward
  bf16_32k           L=32768,  Hq=16, d=128, Hi=8, di=64,  k=512, bf16, fwd+bwd
  bf16_128k_needle   L=131072, Hq=16, d=128, Hi=8, di=64,  k=512, bf16, fwd+bwd,
                     indexer chunk 8192, 10% "needle" tokens
  bf16_256k          L=262144, Hq=32, d=128, Hi=8, di=128, k=512, bf16, fwd+bwd,
                     indexer chunk 4096
  bf16_1m_ties       L=1048576,Hq=16, d=128, Hi=8, di=64,  k=512, bf16, forward,
                     indexer chunk 4096, indexer inputs in {-1,0,1}

Draw order per workload (fixed): Q, K, V, q_I, k_I, w, dO, needle.  Each
tensor has its own torch.Generator seeded from (workload seed, tensor slot),
so drawing a subset of tensors does not change the others.
"""
from __future__ import annotations

import dataclasses
import math

import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    L: int
    Hq: int
    d: int
    Hi: int
    di: int
    k: int
    q_chunk: int
    dtype: str          # "fp32" or "bf16"
    passes: str         # "fwd" or "fwd+bwd"
    seed: int
    indexer: str        # "int3": integers in [-3,3]; "int1": integers in [-1,1]; "normal": N(0,1)
    weights: str        # "int1_4": integers in [1,4]; "pm1": integers in [-1,1]; "uniform01"
    needle: float = 0.0  # fraction of tokens given the shared needle direction

    @property
    def P(self) -> int:
        return self.L // 4

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)

    def with_(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)

    def integer_twin(self) -> "Workload":
        """Same shapes, indexer inputs drawn as small integers so fp32 scores are exact.

        With a needle, the twin's indexer needle is an integer vector as well
        (see make()), so the heavy-tailed selection structure is kept."""
        return self.with_(name=self.name + "_int", indexer="int3", weights="int1_4")


WORKLOADS = {
    "tiny_fp32_fwd": Workload("tiny_fp32_fwd", 4096, 8, 64, 4, 64, 64, 4096, "fp32", "fwd", 0, "int3", "int1_4"),
    "bf16_32k": Workload("bf16_32k", 32768, 16, 128, 8, 64, 512, 8192, "bf16", "fwd+bwd", 1, "normal", "uniform01"),
    "bf16_128k_needle": Workload("bf16_128k_needle", 131072, 16, 128, 8, 64, 512, 8192, "bf16", "fwd+bwd", 2,
                                 "normal", "uniform01", needle=0.10),
    "bf16_256k": Workload("bf16_256k", 262144, 32, 128, 8, 128, 512, 4096, "bf16", "fwd+bwd", 3, "normal", "uniform01"),
    "bf16_1m_ties": Workload("bf16_1m_ties", 1048576, 16, 128, 8, 64, 512, 4096, "bf16", "fwd", 4, "int1", "pm1"),
}

_SLOTS = {"Q": 0, "K": 1, "V": 2, "q_I": 3, "k_I": 4, "w": 5, "dO": 6, "needle": 7}
_CHUNK = 1 << 24  # elements drawn per generator call (bounds host memory)


def _gen(wl: Workload, slot: str) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(1_000_003 * (wl.seed + 1) + 7919 * _SLOTS[slot] + (wl.L % 1_000_033))
    return g


def _torch_dtype(wl: Workload) -> torch.dtype:
    return torch.float32 if wl.dtype == "fp32" else torch.bfloat16


def _draw(shape, kind: str, g: torch.Generator, out_dtype: torch.dtype, add=None, pin=False) -> torch.Tensor:
    """Draw `shape` in chunks of rows; `add(row0, block_fp32)` may modify each block before the cast."""
    out = torch.empty(shape, dtype=out_dtype, pin_memory=pin)
    rows = shape[0]
    per_row = int(math.prod(shape[1:])) if len(shape) > 1 else 1
    step = max(1, _CHUNK // per_row)
    for r0 in range(0, rows, step):
        r1 = min(rows, r0 + step)
        bshape = (r1 - r0,) + tuple(shape[1:])
        if kind == "normal":
            blk = torch.randn(bshape, generator=g, dtype=torch.float32)
        elif kind == "uniform01":
            blk = torch.rand(bshape, generator=g, dtype=torch.float32)
        elif kind == "int3":
            blk = torch.randint(-3, 4, bshape, generator=g, dtype=torch.int32).to(torch.float32)
        elif kind in ("int1", "pm1"):
            blk = torch.randint(-1, 2, bshape, generator=g, dtype=torch.int32).to(torch.float32)
        elif kind == "int1_4":
            blk = torch.randint(1, 5, bshape, generator=g, dtype=torch.int32).to(torch.float32)
        else:
            raise ValueError(kind)
        if add is not None:
            add(r0, blk)
        out[r0:r1] = blk.to(out_dtype)
    return out


def needle_plan(wl: Workload):
    """Needle token mask [L] (bool) and the two shared unit directions (width d and di)."""
    g = _gen(wl, "needle")
    n = int(round(wl.needle * wl.L))
    perm = torch.randperm(wl.L, generator=g)
    mask = torch.zeros(wl.L, dtype=torch.bool)
    mask[perm[:n]] = True
    u_att = torch.randn(wl.d, generator=g, dtype=torch.float64)
    u_idx = torch.randn(wl.di, generator=g, dtype=torch.float64)
    u_att = (u_att / u_att.norm()).to(torch.float32)
    u_idx = (u_idx / u_idx.norm()).to(torch.float32)
    return mask, u_att, u_idx


def make(wl: Workload, tensors=("Q", "K", "V", "q_I", "k_I", "w", "dO"), pin: bool = False) -> dict:
    """Host (CPU) tensors for the workload, in the layer's dtypes.

    Q [L,Hq,d], K [L,d], V [L,d], dO [L,Hq,d] and q_I [L,Hi,di], k_I [L,di] in
    the layer dtype; w [L,Hi] fp32.  With a needle fraction, every needle
    token gets 4*sqrt(width)*u added (before the cast) to Q (all heads), K,
    q_I (all heads) and k_I, with one shared unit vector u per width.  When
    the indexer inputs are integers (an integer twin), the indexer's needle
    is the integer vector 3*sign(u) instead, so q_I and k_I stay integers
    (|q_I| <= 6, |kpool| <= 24) and every fp32 score stays exact.
    """
    dt = _torch_dtype(wl)
    mask = u_att = u_idx = None
    if wl.needle > 0:
        mask, u_att, u_idx = needle_plan(wl)

    def needle_add(u, width, integer=False):
        if mask is None:
            return None
        amp = 4.0 * math.sqrt(width)
        if integer:
            u = 3.0 * torch.sign(u)
            amp = 1.0

        def add(r0, blk):
            m = mask[r0:r0 + blk.shape[0]]
            if blk.dim() == 3:
                blk[m] += amp * u.view(1, 1, -1)
            else:
                blk[m] += amp * u.view(1, -1)
        return add

    out = {}
    for name in tensors:
        g = _gen(wl, name)
        if name == "Q":
            out[name] = _draw((wl.L, wl.Hq, wl.d), "normal", g, dt, needle_add(u_att, wl.d), pin)
        elif name == "K":
            out[name] = _draw((wl.L, wl.d), "normal", g, dt, needle_add(u_att, wl.d), pin)
        elif name == "V":
            out[name] = _draw((wl.L, wl.d), "normal", g, dt, None, pin)
        elif name == "dO":
            out[name] = _draw((wl.L, wl.Hq, wl.d), "normal", g, dt, None, pin)
        elif name == "q_I":
            out[name] = _draw((wl.L, wl.Hi, wl.di), wl.indexer, g, dt,
                              needle_add(u_idx, wl.di, wl.indexer != "normal"), pin)
        elif name == "k_I":
            out[name] = _draw((wl.L, wl.di), wl.indexer, g, dt, needle_add(u_idx, wl.di, wl.indexer != "normal"), pin)
        elif name == "w":
            out[name] = _draw((wl.L, wl.Hi), wl.weights, g, torch.float32, None, pin)
        else:
            raise ValueError(name)
    return out


def sample_rows(wl: Workload, n: int = 1024, seed: int = 12345):
    """Seeded query rows for sampled parity checks: the first 8 rows, every
    indexer-chunk boundary +-1, the last 8 rows, and uniform draws to reach n."""
    L, C = wl.L, wl.q_chunk
    rows = set(range(min(8, L)))
    rows.update(range(max(0, L - 8), L))
    for b in range(C, L, C):
        rows.update((b - 1, b, b + 1))
    g = torch.Generator().manual_seed(seed + wl.seed)
    extra = torch.randint(0, L, (max(0, n - len(rows)) * 2,), generator=g).tolist()
    for r in extra:
        if len(rows) >= n:
            break
        rows.add(int(r))
    return sorted(r for r in rows if 0 <= r < L)


def to_f32_numpy(t: torch.Tensor):
    """Exact fp32 copy of a host tensor (bf16 values are exact in fp32)."""
    return t.to(torch.float32).numpy()
