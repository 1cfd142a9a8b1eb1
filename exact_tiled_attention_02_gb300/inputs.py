"""Seeded synthetic inputs shared by the tests, the bench and the oracle
checks.  Holds no attention arithmetic: it only draws numbers.

Recipe: a CPU ``torch.Generator`` seeded with ``seed``; q, k, v and (if asked)
dO are drawn in that order as float32 standard normals of shape [B, H, N, d];
q and k are multiplied by ``qk_mult``; everything is then cast to the
workload's dtype (bf16 rounding to nearest even).  The oracle receives the
cast values widened to float64, so both sides see identical inputs.
"""

from __future__ import annotations

import torch

DTYPES = {"f32": torch.float32, "bf16": torch.bfloat16}


def make_inputs(B: int, H: int, N: int, d: int, dtype: str = "bf16", seed: int = 0, qk_mult: float = 1.0,
                with_do: bool = False):
    g = torch.Generator().manual_seed(seed)
    shape = (B, H, N, d)
    q = torch.randn(shape, generator=g, dtype=torch.float32)
    k = torch.randn(shape, generator=g, dtype=torch.float32)
    v = torch.randn(shape, generator=g, dtype=torch.float32)
    do = torch.randn(shape, generator=g, dtype=torch.float32) if with_do else None
    if qk_mult != 1.0:
        q.mul_(qk_mult)
        k.mul_(qk_mult)
    t = DTYPES[dtype]
    out = [q.to(t), k.to(t), v.to(t)]
    if with_do:
        out.append(do.to(t))
    return tuple(out)


def workload_inputs(w, with_do: bool = False):
    """Inputs of a ``configs.Workload`` (seed = workload index - 1)."""
    return make_inputs(w.B, w.H, w.N, w.d, w.dtype, w.seed, w.qk_mult, with_do)
