"""Seeded synthetic inputs and the named workloads of the all-gather matmul.

This module is shared by the CUDA path's tests and benchmark and by the CPU
oracle's tests.  It holds no arithmetic of the method itself: it only draws
random shards ``X_r`` and the right-hand side ``Y`` and records the workload
shapes.  Both sides receive exactly the same tensors.

Recipe (one reading of the workloads, stated once here):

* A CPU ``torch.Generator`` seeded with ``seed`` (0 unless stated) draws, in
  this order, ``X_0 .. X_{P-1}`` (each ``[m_per_device, k]``) and then ``Y``.
* Values are drawn in float32 and rounded to bfloat16 (or, for the fp16
  variant, float16) by PyTorch's round-to-nearest-even cast.
* ``Y`` is drawn directly in its stored layout: ``[k, n]`` when
  ``rhs_transpose`` is false, ``[n, k]`` when it is true (the flag of the
  Pallas TPU kernel's ``all_gather_matmul`` API).
* "uniform" means U[-1, 1); "normal" means X ~ N(0, 1) and Y ~ N(0, 0.02**2)
  (0.02 read as the standard deviation).

The pages name no public dataset or benchmark suite; these synthetic tensors
stand in for the workloads they describe.
"""
from __future__ import annotations

import dataclasses
from typing import List, Tuple

import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    """One problem instance: P shards of ``[m_per_device, k]`` times ``Y``."""

    name: str
    P: int
    m_per_device: int
    k: int
    n: int
    rhs_transpose: bool
    my_id: int
    dist: str = "normal"  # "normal" or "uniform"
    seed: int = 0

    @property
    def M(self) -> int:
        return self.P * self.m_per_device

    @property
    def flops(self) -> int:
        """2*M*k*n, the cost model of the Pallas kernel's CostEstimate."""
        return 2 * self.M * self.k * self.n

    @property
    def unique_bytes(self) -> int:
        """bf16 bytes of gathered X, Y and O, each moved once."""
        return 2 * (self.M * self.k + self.k * self.n + self.M * self.n)


def _sweep() -> List[Workload]:
    out = []
    for P in (2, 4, 8):
        for m in (8, 32, 128, 1000, 4096):
            for rt in (False, True):
                out.append(Workload(f"sweep_P{P}_m{m}_{'rt' if rt else 'nt'}", P, m, 5120,
                                    2560, rt, P - 1))
    return out


# The five workload families: a tiny uniform case, a decode-like Y-read-bound
# case, a mid-size case, a prefill-like compute-bound case, and a sweep.
WORKLOADS = {
    "c1_tiny": Workload("c1_tiny", 2, 16, 256, 128, False, 0, "uniform"),
    "c2_decode": Workload("c2_decode", 4, 64, 4096, 1024, True, 1),
    "c3_mid": Workload("c3_mid", 8, 256, 8192, 3584, False, 3),
    "c4_prefill": Workload("c4_prefill", 8, 2048, 8192, 7168, True, 5),
    # the prefill workload with a quarter of its rows: small enough for a
    # full ncu capture of the row-tile kernel, still larger than L2
    "c4_quarter": Workload("c4_quarter", 8, 512, 8192, 7168, True, 5),
}
SWEEP = _sweep()
for _w in SWEEP:
    WORKLOADS[_w.name] = _w


def make_inputs(P: int, m_per_device: int, k: int, n: int, rhs_transpose: bool,
                dist: str = "normal", seed: int = 0, y_std: float = 0.02, dtype: str = "bf16"
                ) -> Tuple[List[torch.Tensor], torch.Tensor]:
    """Draw the P shards and ``Y`` on the CPU (see module recipe); ``dtype``
    "bf16" or "f16" is the type the float32 draws are rounded to."""
    tdt = {"bf16": torch.bfloat16, "f16": torch.float16}[dtype]
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    xs = []
    for _ in range(P):
        if dist == "uniform":
            x = torch.rand((m_per_device, k), generator=g, dtype=torch.float32) * 2.0 - 1.0
        elif dist == "normal":
            x = torch.randn((m_per_device, k), generator=g, dtype=torch.float32)
        else:
            raise ValueError(f"unknown distribution {dist!r}")
        xs.append(x.to(tdt))
    yshape = (n, k) if rhs_transpose else (k, n)
    if dist == "uniform":
        y = torch.rand(yshape, generator=g, dtype=torch.float32) * 2.0 - 1.0
    else:
        y = torch.randn(yshape, generator=g, dtype=torch.float32) * y_std
    return xs, y.to(tdt)


def make_workload_inputs(w: Workload) -> Tuple[List[torch.Tensor], torch.Tensor]:
    return make_inputs(w.P, w.m_per_device, w.k, w.n, w.rhs_transpose, w.dist, w.seed)
