"""The five attention workloads: shapes, dtypes, value scaling and masks.

Each entry states a problem, not an algorithm: B batches x H heads of
length-N sequences with head dimension d; ``qk_mult`` multiplies the standard
normal Q and K draws (8 makes the running-max rescale work hard: scaled logits
with a standard deviation of about 64); ``window`` is the full width of the
symmetric local window (0 = unmasked); ``passes`` says which passes the
workload exercises.
"""

from __future__ import annotations

import math
from dataclasses import dataclass


@dataclass(frozen=True)
class Workload:
    index: int
    name: str
    B: int
    H: int
    N: int
    d: int
    dtype: str  # "f32" or "bf16"
    window: int = 0
    qk_mult: float = 1.0
    passes: tuple = ("fwd",)

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)

    @property
    def seed(self) -> int:
        return self.index - 1

    def pairs_per_head(self) -> int:
        """Number of (query, key) pairs that take part in the softmax."""
        if self.window <= 0:
            return self.N * self.N
        r = (self.window - 1) // 2
        n = self.N
        # sum over i of |{j : |i - j| <= r, 0 <= j < n}|
        return sum(min(n - 1, i + r) - max(0, i - r) + 1 for i in range(n)) if n <= 4096 else \
            (2 * r + 1) * n - r * (r + 1)

    def fwd_flops(self) -> float:
        """4 * B * H * N^2 * d, scaled by the fraction of unmasked pairs."""
        return 4.0 * self.B * self.H * self.d * self.pairs_per_head()

    def bwd_flops(self) -> float:
        return 2.5 * self.fwd_flops()


WORKLOADS = {
    1: Workload(1, "fwd_f32_b1_h1_n6_d4", 1, 1, 6, 4, "f32"),
    2: Workload(2, "fwd_bf16_b4_h16_n2048_d64", 4, 16, 2048, 64, "bf16"),
    3: Workload(3, "fwd_bf16_b2_h16_n8192_d128_qk8", 2, 16, 8192, 128, "bf16", qk_mult=8.0),
    4: Workload(4, "fwd_bf16_b1_h32_n16384_d128_w257", 1, 32, 16384, 128, "bf16", window=257),
    5: Workload(5, "bwd_bf16_b4_h16_n4096_d128", 4, 16, 4096, 128, "bf16", passes=("fwd", "bwd")),
}


def custom_workload(spec: str, dtype: str = "bf16") -> Workload:
    """A workload of another shape, from ``"B,H,N,d[,window[,qk_mult]]"``, in
    ``dtype`` ("bf16" or "f32").  It has index 0, so its inputs are drawn with
    seed -1."""
    if dtype not in ("bf16", "f32"):
        raise ValueError("dtype must be bf16 or f32")
    parts = [p.strip() for p in spec.split(",")]
    if not 4 <= len(parts) <= 6:
        raise ValueError("shape must be B,H,N,d[,window[,qk_mult]]")
    B, H, N, d = (int(x) for x in parts[:4])
    window = int(parts[4]) if len(parts) > 4 else 0
    qk = float(parts[5]) if len(parts) > 5 else 1.0
    name = f"custom_{dtype}_b{B}_h{H}_n{N}_d{d}" + (f"_w{window}" if window > 0 else "") + \
        (f"_qk{qk:g}" if qk != 1.0 else "")
    return Workload(0, name, B, H, N, d, dtype, window=window, qk_mult=qk, passes=("fwd", "bwd"))
