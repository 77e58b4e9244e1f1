"""Seeded synthetic inputs for Evoformer attention.

This module only draws random numbers and builds masks; it holds none of the
attention arithmetic.  Both the CUDA path and the CPU oracle consume the
tensors it returns (the oracle upcasts the dtype-rounded values exactly).

Workloads follow the shapes of the four usages on the web page
"DeepSpeed4Science 技术指南：AI4Science 大模型长序列训练与 Evoformer 内存高效
注意力内核实战" (§3.6: MSA row-wise with pair bias, MSA column-wise with the
mask only, triangle attention with the edge bias) and the test shapes named
in its §3.5, (1, 256, 256, 4, 32) and (1, 512, 256, 8, 8).

Recipe (the page gives no data; these are the stated synthetic readings):

* Q, K, V, dO ~ N(0, 1), drawn in float32 from ``numpy.random.default_rng``
  in the fixed order Q, K, V, dO, mask, pair bias; then rounded to the input
  dtype (round to nearest even).
* Key mask ``bias1`` [B, N, 1, 1, L]: 0 for kept keys and -1e9 for masked
  keys, rounded to the dtype (fp16 gives -inf, bf16 gives -998244352).
  ``("random", f)``: every (b, n) row masks exactly round(f*L) keys chosen by
  a per-row random permutation (at least one key stays).  ``("tail", f)``:
  keys j >= L - round(f*L) are masked in every row.
* Pair bias ``bias2`` [B, 1, H, L, L] ~ N(0, sigma^2) or absent.
"""

from __future__ import annotations

from dataclasses import dataclass, field
from typing import Optional, Tuple

import numpy as np
import torch

MASK_VALUE = -1.0e9

DTYPES = {"fp16": torch.float16, "bf16": torch.bfloat16}


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    N: int
    L: int
    H: int
    D: int
    dtypes: Tuple[str, ...]
    mask: Optional[Tuple[str, float]]
    bias2_sigma: Optional[float]
    what: str = field(default="", compare=False)

    @property
    def shape(self):
        return (self.B, self.N, self.L, self.H, self.D)


WORKLOADS = {
    "tiny": Workload("tiny", 1, 8, 32, 2, 16, ("fp16",), ("random", 0.10), 1.0,
                     "tiny CPU-checkable instance"),
    "msa_row": Workload("msa_row", 1, 256, 256, 4, 32, ("fp16", "bf16"),
                        ("random", 0.05), 1.0,
                        "MSA row-wise attention with pair bias"),
    "many_head": Workload("many_head", 1, 512, 256, 8, 8, ("bf16",),
                          ("random", 0.05), 0.5,
                          "many-head small-D row attention"),
    "msa_col": Workload("msa_col", 1, 384, 1024, 8, 32, ("bf16",),
                        ("tail", 0.15), None,
                        "MSA column-wise attention, mask only"),
    "triangle": Workload("triangle", 1, 512, 512, 4, 32, ("bf16",),
                         ("tail", 0.03), 1.0,
                         "triangle attention over the pair representation"),
}


def masked_count(L: int, frac: float) -> int:
    """Number of masked keys per row: round(frac * L), leaving one key kept."""
    return int(min(max(round(frac * L), 0), max(L - 1, 0)))


def make_inputs(B, N, L, H, D, dtype="bf16", mask=("random", 0.05),
                bias2_sigma=1.0, seed=0, has_bias1=True):
    """Return a dict of CPU torch tensors in ``dtype``:
    q, k, v, do [B,N,L,H,D]; bias1 [B,N,1,1,L] or None; bias2 [B,1,H,L,L] or None.
    """
    tdt = DTYPES[dtype]
    rng = np.random.default_rng(seed)
    shp = (B, N, L, H, D)

    def normal(shape, sigma=1.0):
        x = rng.standard_normal(size=shape, dtype=np.float32)
        if sigma != 1.0:
            x *= np.float32(sigma)
        return torch.from_numpy(x).to(tdt)

    q = normal(shp)
    k = normal(shp)
    v = normal(shp)
    do = normal(shp)

    bias1 = None
    if has_bias1 and mask is not None:
        kind, frac = mask
        m = np.zeros((B, N, 1, 1, L), dtype=np.float32)
        cnt = masked_count(L, frac)
        if kind == "random":
            for b in range(B):
                for n in range(N):
                    idx = rng.permutation(L)[:cnt]
                    m[b, n, 0, 0, idx] = MASK_VALUE
        elif kind == "tail":
            if cnt > 0:
                m[..., L - cnt:] = MASK_VALUE
        else:
            raise ValueError(f"unknown mask kind {kind!r}")
        bias1 = torch.from_numpy(m).to(tdt)
    elif has_bias1:
        bias1 = torch.zeros((B, N, 1, 1, L), dtype=tdt)

    bias2 = None
    if bias2_sigma is not None:
        bias2 = normal((B, 1, H, L, L), bias2_sigma)

    return {"q": q, "k": k, "v": v, "do": do, "bias1": bias1, "bias2": bias2}


def workload_inputs(name: str, dtype: Optional[str] = None, seed: int = 0):
    w = WORKLOADS[name]
    dt = dtype or w.dtypes[-1]
    return make_inputs(*w.shape, dtype=dt, mask=w.mask,
                       bias2_sigma=w.bias2_sigma, seed=seed)
