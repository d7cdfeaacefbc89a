"""Workload definitions and seeded synthetic inputs.

This module holds the five benchmark workloads (grid sizes, basis, cutoff,
batch and channel counts, dtype, seed) and the seeded input generators.  It
contains none of the method's arithmetic, so both the CUDA path and the CPU
oracle draw their inputs from it.

Inputs are drawn with a CPU ``torch.Generator`` seeded per workload, in fp32
with ``torch.randn``, in the fixed order x, W, dy, G (each only when the
workload uses it), then cast with round-to-nearest-even to the workload dtype.
W is drawn N(0, 1) and scaled by 1/sqrt(Cin*K), i.e. variance 1/(Cin*K).
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch

ISO, ANISO = 0, 1


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    C: int
    Cout: int | None
    grid_in: tuple       # (nlat, nlon, poles)
    grid_out: tuple
    kind: int            # ISO or ANISO
    nrad: int            # radial hats
    cutoff: float        # radians
    dtype: str           # "f32" or "bf16"
    seed: int
    ops: tuple = field(default=())

    @property
    def K(self) -> int:
        return self.nrad if self.kind == ISO else 3 * self.nrad

    @property
    def torch_dtype(self):
        return torch.float32 if self.dtype == "f32" else torch.bfloat16

    def shapes(self):
        Hin, Win = self.grid_in[:2]
        Hout, Wout = self.grid_out[:2]
        s = {
            "x": (self.B, self.C, Hin, Win),
            "X": (self.B, self.C, self.K, Hout, Wout),
        }
        if self.Cout is not None:
            s["W"] = (self.Cout, self.C, self.K)
            s["y"] = (self.B, self.Cout, Hout, Wout)
        return s


WORKLOADS = {
    w.name: w
    for w in [
        Workload("tiny_f32_16x32", 1, 2, None, (16, 32, 0), (16, 32, 0), ISO, 3,
                 2 * math.pi / 16, "f32", 0, ("fwd", "bwd")),
        Workload("iso5_bf16_64x128", 4, 32, None, (64, 128, 0), (64, 128, 0), ISO, 5,
                 3 * math.pi / 64, "bf16", 1, ("fwd", "bwd")),
        Workload("down_fused_128x256_to_64x128", 8, 64, 64, (128, 256, 0), (64, 128, 0), ANISO,
                 3, 3 * math.pi / 64, "bf16", 2, ("fused",)),
        Workload("fused_bwd_361x720", 2, 128, 128, (361, 720, 1), (361, 720, 1), ANISO, 3,
                 4 * math.pi / 360, "bf16", 3, ("fused", "fused_bwd")),
        Workload("down_fused_bwd_721x1440_to_361x720", 1, 256, 256, (721, 1440, 1),
                 (361, 720, 1), ANISO, 3, 3 * math.pi / 360, "bf16", 4,
                 ("fused", "fused_bwd")),
    ]
}

ORDER = list(WORKLOADS)
LARGEST = ORDER[-1]

# The benchmark shapes the DISCO Kernel Development Guide lists (§Profiling /
# Serial Benchmarks: 256 and 512 channels on 360 x 720, and 80 -> 512
# channels from 721 x 1440 to 360 x 720), on Legendre-Gauss grids (poles = 2)
# with theta_cutoff = 0.017 and kernel_shape (3, 3).  The page's "harmonic" basis and "mean" normalisation
# are not defined there; this library's anisotropic basis (3 radial hats x
# {1, cos, sin}, K = 9) and per-ring normalisation stand in.  B is not given:
# 1.  The 721-row equiangular input includes the poles.  Parity-test cases,
# not benchmark lines.
PAGE_WORKLOADS = {
    w.name: w
    for w in [
        Workload("page_self_256x360x720_gauss", 1, 256, 256, (360, 720, 2), (360, 720, 2), ANISO, 3,
                 0.017, "bf16", 5, ("fused", "fused_bwd")),
        Workload("page_self_512x360x720_gauss", 1, 512, 512, (360, 720, 2), (360, 720, 2), ANISO, 3,
                 0.017, "bf16", 7, ("fused", "fused_bwd")),
        Workload("page_down_80x721x1440_to_360x720_gauss", 1, 80, 512, (721, 1440, 1), (360, 720, 2),
                 ANISO, 3, 0.017, "bf16", 6, ("fwd", "bwd", "fused", "fused_bwd")),
    ]
}


def make_inputs(w: Workload, with_G: bool = False, device="cpu") -> dict:
    """Seeded inputs of workload ``w`` as CPU tensors in ``w``'s dtype.

    x ~ N(0,1); W ~ N(0, 1/(Cin*K)) (fused workloads); dy ~ N(0,1) (fused
    workloads); G ~ N(0,1) of the contraction output shape (workloads that run
    the plain transpose, or when ``with_G``)."""
    g = torch.Generator(device="cpu")
    g.manual_seed(w.seed)
    dt = w.torch_dtype
    sh = w.shapes()
    out = {"x": torch.randn(sh["x"], generator=g, dtype=torch.float32).to(dt)}
    if w.Cout is not None:
        Wf = torch.randn(sh["W"], generator=g, dtype=torch.float32) / math.sqrt(w.C * w.K)
        out["W"] = Wf.to(dt)
        out["dy"] = torch.randn(sh["y"], generator=g, dtype=torch.float32).to(dt)
    if "bwd" in w.ops or with_G:
        out["G"] = torch.randn(sh["X"], generator=g, dtype=torch.float32).to(dt)
    if device != "cpu":
        out = {k: v.to(device) for k, v in out.items()}
    return out


def sample_points(shape, n: int, seed: int, include_corners: bool = True):
    """n seeded index tuples into ``shape`` (plus the first and last element)."""
    g = torch.Generator(device="cpu")
    g.manual_seed(10_000 + seed)
    cols = [torch.randint(0, d, (n,), generator=g) for d in shape]
    pts = torch.stack(cols, 1)
    if include_corners:
        first = torch.zeros(1, len(shape), dtype=torch.int64)
        last = torch.tensor([[d - 1 for d in shape]], dtype=torch.int64)
        pts = torch.cat([first, last, pts], 0)
    return pts
