"""Seeded synthetic workloads for HSTU attention.

This module draws inputs only: sequence lengths, packed q/k/v/dO tensors and
cumulative lengths.  It holds none of the attention arithmetic, so both the
CUDA path's tests and the CPU oracle can be fed from it.

Workloads stand in for recommender user histories ("HSTU Attention (Blackwell
SM100/SM103)": packed THD tensors, section "Tensor layout"); no dataset is
involved.  Recipe for every workload:

* ``torch.Generator('cpu').manual_seed(seed)`` (seed 0 by default);
* draw order: sequence lengths, then q, k, v, dO;
* values are fp32 normal samples times ``std``, rounded to bf16 or fp16
  (round to nearest even), on the host;
* ``cu_seqlens_q == cu_seqlens_k`` (int32, leading 0), ``max_seqlen`` is the
  largest drawn length, ``scaling_seqlen`` is ``max_seqlen`` unless fixed.

Length laws:
* ``uniform``: integers uniform on [lo, hi], both ends included;
* ``powerlaw``: density proportional to L**-a on [lo, hi], drawn by inverse
  CDF and floored, clamped to [lo, hi];
* ``fixed``: every sequence has length ``lo``.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional, Sequence

import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    batch: int
    length_law: str              # "list" | "uniform" | "powerlaw" | "fixed"
    heads: int
    head_dim: int
    dtype: torch.dtype
    alpha: float
    causal: bool
    std: float = 1.0
    lo: int = 0
    hi: int = 0
    exponent: float = 0.0
    lengths: Optional[Sequence[int]] = None
    scaling_seqlen: Optional[int] = None   # None -> max_seqlen_q

    def describe(self) -> dict:
        law = {"list": f"lengths {list(self.lengths or [])}",
               "uniform": f"uniform integers [{self.lo},{self.hi}]",
               "powerlaw": f"truncated power law exponent {self.exponent} on [{self.lo},{self.hi}]",
               "fixed": f"all {self.lo}"}[self.length_law]
        return {"workload": self.name, "B": self.batch, "lengths": law,
                "H": self.heads, "D": self.head_dim,
                "dtype": str(self.dtype).replace("torch.", ""),
                "alpha": self.alpha, "mask": "causal" if self.causal else "full",
                "values": f"N(0,{self.std}^2) rounded to dtype, seed 0",
                "scaling_seqlen": self.scaling_seqlen or "max_seqlen_q"}


WORKLOADS = {
    # tiny case: four packed sequences, fixed lengths
    "tiny": Workload("tiny", 4, "list", 2, 64, torch.bfloat16, 1.0 / math.sqrt(64),
                     True, lengths=(17, 64, 100, 128), scaling_seqlen=128),
    # recommender training batch
    "recsys": Workload("recsys", 32, "uniform", 4, 128, torch.bfloat16,
                       1.0 / math.sqrt(128), True, lo=256, hi=1024),
    # long user histories
    "long": Workload("long", 8, "uniform", 4, 128, torch.bfloat16,
                     1.0 / math.sqrt(128), True, lo=2048, hi=8192),
    # heavily skewed ragged batch
    "skewed": Workload("skewed", 128, "powerlaw", 8, 64, torch.float16,
                       1.0 / math.sqrt(64), True, std=0.5, lo=16, hi=4096,
                       exponent=1.5),
    # full (non-causal) mask, long fixed sequences
    "full": Workload("full", 16, "fixed", 2, 256, torch.float16, 1.0 / 16.0,
                     False, lo=4096, scaling_seqlen=4096),
}


def draw_lengths(w: Workload, gen: torch.Generator) -> list:
    if w.length_law == "list":
        return [int(x) for x in w.lengths]
    if w.length_law == "fixed":
        return [int(w.lo)] * w.batch
    if w.length_law == "uniform":
        return [int(x) for x in torch.randint(w.lo, w.hi + 1, (w.batch,), generator=gen)]
    if w.length_law == "powerlaw":
        u = torch.rand(w.batch, generator=gen, dtype=torch.float64)
        e = 1.0 - w.exponent                   # CDF ~ L**e, e < 0 here
        a, b = float(w.lo) ** e, float(w.hi) ** e
        L = torch.floor((a + u * (b - a)) ** (1.0 / e))
        return [int(x) for x in L.clamp(w.lo, w.hi)]
    raise ValueError(w.length_law)


def cu_seqlens(lengths: Sequence[int]) -> torch.Tensor:
    cu = [0]
    for L in lengths:
        cu.append(cu[-1] + int(L))
    return torch.tensor(cu, dtype=torch.int32)


def make_inputs(w: Workload, seed: int = 0, lengths: Optional[Sequence[int]] = None,
                with_grad: bool = True) -> dict:
    """Host (CPU) inputs of workload ``w`` drawn from ``seed``.

    ``lengths`` overrides the length law (the values are still drawn from the
    same generator after the lengths would have been drawn).
    """
    gen = torch.Generator(device="cpu").manual_seed(seed)
    drawn = draw_lengths(w, gen)
    lens = list(lengths) if lengths is not None else drawn
    T = int(sum(lens))
    H, D = w.heads, w.head_dim

    def draw():
        return (torch.randn(T, H, D, generator=gen) * w.std).to(w.dtype)

    q, k, v = draw(), draw(), draw()
    do = draw() if with_grad else None
    cu = cu_seqlens(lens)
    max_seqlen = max(lens) if lens else 0
    return {"q": q, "k": k, "v": v, "do": do, "cu_seqlens_q": cu,
            "cu_seqlens_k": cu.clone(), "max_seqlen_q": max_seqlen,
            "max_seqlen_k": max_seqlen, "lengths": lens,
            "alpha": w.alpha, "causal": w.causal,
            "scaling_seqlen": w.scaling_seqlen, "workload": w}


def random_inputs(lengths_q: Sequence[int], lengths_k: Sequence[int], H: int, D: int,
                  dtype: torch.dtype, seed: int, std: float = 1.0) -> dict:
    """Generic seeded THD inputs for arbitrary (possibly unequal) q/k lengths."""
    gen = torch.Generator(device="cpu").manual_seed(seed)
    Tq, Tk = int(sum(lengths_q)), int(sum(lengths_k))

    def draw(T):
        return (torch.randn(T, H, D, generator=gen) * std).to(dtype)

    q, k, v, do = draw(Tq), draw(Tk), draw(Tk), draw(Tq)
    return {"q": q, "k": k, "v": v, "do": do,
            "cu_seqlens_q": cu_seqlens(lengths_q), "cu_seqlens_k": cu_seqlens(lengths_k),
            "max_seqlen_q": max(lengths_q) if len(lengths_q) else 0,
            "max_seqlen_k": max(lengths_k) if len(lengths_k) else 0}
