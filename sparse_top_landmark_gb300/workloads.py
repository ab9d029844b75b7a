"""Seeded synthetic inputs for the MiTA forward pass.

This module only draws numbers: it holds none of the method's arithmetic and is
shared, unchanged, by the CPU oracle's tests, the GPU parity tests, ``smoke()``
and ``bench.py``.

Recipe (one per named workload, all tensors row-major ``[B, H, N, d]``):

* ``iid``: Q and K are i.i.d. N(0, 1).
* ``mixture``: per (batch, head) ``C`` cluster centres are drawn from N(0, I_d);
  every token ``t`` draws one cluster ``c_t`` uniformly; then
  ``q_t = mu[c_t] + sigma * eps`` and ``k_t = mu[c_t] + sigma * eps'`` with
  independent noise and a shared assignment.
* V is always i.i.d. N(0, 1).
* Draws are float32 from a CPU ``torch.Generator`` seeded with
  ``seed + 1000 * index`` (index = the workload's position in ``WORKLOADS``),
  then rounded once (round-to-nearest-even) to the workload's dtype.

The shapes follow the pages' experiments: a DeiT-S image grid (ImageNet-1K
stand-in, MiTA tutorial ch. 7 table 2: m = k = 25), an ADE20K-sized grid
(tutorial ch. 7 table 4: m = k = 49, 98 entries per query) and the two long
synthetic sequences of the throughput figure (tutorial ch. 7 figure 5:
m * k ~= N / 4 at 64K and 1024K tokens).
"""
from __future__ import annotations

from dataclasses import dataclass, asdict
from typing import Optional

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    N: int
    d: int
    dtype: str          # "f32" or "bf16"
    grid_h: int         # grid_h == 1: 1D sequence pooled to m contiguous windows
    grid_w: int
    m: int
    topk: int
    s: int
    qk: str             # "iid" or "mixture"
    clusters: int = 0
    sigma: float = 0.0
    index: int = 0

    @property
    def queries(self) -> int:
        return self.B * self.H * self.N

    @property
    def torch_dtype(self) -> torch.dtype:
        return torch.float32 if self.dtype == "f32" else torch.bfloat16

    def as_dict(self) -> dict:
        return asdict(self)


WORKLOADS = {
    w.name: w
    for w in [
        Workload("tiny_1d", 1, 1, 64, 16, "f32", 1, 64, 4, 4, 1, "iid", index=0),
        Workload("vit_s_14x14", 64, 6, 196, 64, "bf16", 14, 14, 25, 25, 1,
                 "mixture", 16, 0.3, index=1),
        Workload("seg_32x32", 16, 6, 1024, 64, "bf16", 32, 32, 49, 49, 1,
                 "mixture", 16, 0.3, index=2),
        Workload("long_64k", 4, 2, 65536, 64, "bf16", 1, 65536, 128, 128, 1,
                 "mixture", 64, 0.3, index=3),
        Workload("long_1m", 1, 2, 1048576, 64, "bf16", 1, 1048576, 512, 512, 1,
                 "mixture", 256, 0.3, index=4),
    ]
}


def custom(name: str, B: int, H: int, N: int, d: int, dtype: str, grid_h: int,
           grid_w: int, m: int, topk: int, s: int = 1, qk: str = "mixture",
           clusters: int = 8, sigma: float = 0.3, index: int = 100) -> Workload:
    """A workload of arbitrary shape (used for ragged and edge-case tests)."""
    return Workload(name, B, H, N, d, dtype, grid_h, grid_w, m, topk, s, qk,
                    clusters, sigma, index)


def make_qkv(w: Workload, seed: int = 0, B: Optional[int] = None,
             H: Optional[int] = None):
    """Return (q, k, v) CPU tensors of dtype ``w.torch_dtype``, shape [B,H,N,d].

    ``B``/``H`` may be given smaller than the workload's to draw only the first
    batches/heads; those draws differ from the full tensor's, so use this only
    where the full workload is never compared.
    """
    B = w.B if B is None else B
    H = w.H if H is None else H
    g = torch.Generator(device="cpu")
    g.manual_seed(seed + 1000 * w.index)
    shape = (B, H, w.N, w.d)
    if w.qk == "iid":
        q = torch.randn(shape, generator=g, dtype=torch.float32)
        k = torch.randn(shape, generator=g, dtype=torch.float32)
    elif w.qk == "mixture":
        C = w.clusters
        mu = torch.randn((B, H, C, w.d), generator=g, dtype=torch.float32)
        assign = torch.randint(0, C, (B, H, w.N), generator=g)
        centre = torch.gather(mu, 2, assign.unsqueeze(-1).expand(B, H, w.N, w.d))
        del assign
        q = torch.randn(shape, generator=g, dtype=torch.float32)
        q.mul_(w.sigma).add_(centre)
        k = torch.randn(shape, generator=g, dtype=torch.float32)
        k.mul_(w.sigma).add_(centre)
        del centre
    else:
        raise ValueError(f"unknown Q/K recipe {w.qk!r}")
    v = torch.randn(shape, generator=g, dtype=torch.float32)
    dt = w.torch_dtype
    if dt != torch.float32:
        q, k, v = q.to(dt), k.to(dt), v.to(dt)
    return q.contiguous(), k.contiguous(), v.contiguous()
