"""disco_fused_conv_bwd_weight (weight gradient of the fused convolution)
against the fp64 oracle: every element on small cases (ragged output-channel,
C*K and pixel tiles, s = 2, pole grids), sampled channels of the largest
workload in the benchmark's shapes, determinism, unsupported shapes."""
import math

import numpy as np
import pytest
import torch

import oracle
from sparse_spherical_convolution_gb300.workloads import WORKLOADS, make_inputs
from tests._helpers import TOL, rel_err, to_np32

pytestmark = pytest.mark.gpu
BF = torch.bfloat16


@pytest.fixture(scope="module")
def lib():
    from sparse_spherical_convolution_gb300 import build
    build.build()
    import sparse_spherical_convolution_gb300 as d
    d.disco_device_status(clear=True)
    return d


# (grid_in, grid_out, kind, nrad, cutoff, B, Cin, Cout)
SMALL = [
    ((33, 64, 1), (33, 64, 1), 1, 3, 3 * math.pi / 32, 2, 64, 48),      # Cout < 128, 3 C*K tiles
    ((64, 128, 0), (64, 128, 0), 0, 5, 3 * math.pi / 64, 1, 32, 16),    # K = 5, C*K = 160
    ((128, 256, 0), (64, 128, 0), 1, 3, 3 * math.pi / 64, 2, 32, 136),  # s = 2, 2 o tiles, C*K = 288
]


def _run(lib, psi, x, dy, B, Cin, Cout):
    K = psi.c.K
    dW = torch.full((Cout, Cin, K), float("nan"), dtype=BF, device="cuda")
    nws = lib.disco_fused_conv_bwd_weight_workspace_bytes(psi.c, B, Cin, Cout)
    assert nws > 0
    ws = torch.empty(nws, dtype=torch.uint8, device="cuda")
    lib.disco_fused_conv_bwd_weight(psi.c, x, dy, dW, B, Cin, Cout, ws)
    return dW


@pytest.mark.parametrize("case", SMALL, ids=lambda c: f"{c[0]}->{c[1]}-B{c[5]}Ci{c[6]}Co{c[7]}")
def test_weight_grad_full_compare(lib, case):
    gi, go, kind, nrad, cut, B, Cin, Cout = case
    ref = oracle.build_psi(gi, go, kind, nrad, cut)
    psi = lib.Psi(gi, go, kind, nrad, cut)
    g = torch.Generator().manual_seed(21)
    x = torch.randn((B, Cin, gi[0], gi[1]), generator=g).to(BF)
    dy = torch.randn((B, Cout, go[0], go[1]), generator=g).to(BF)
    xd, dyd = x.cuda(), dy.cuda()
    dW = _run(lib, psi, xd, dyd, B, Cin, Cout)
    torch.cuda.synchronize()
    assert lib.disco_device_status() == 0
    assert not torch.isnan(dW).any()
    want, S = oracle.fused_bwd_weight(ref, to_np32(x), to_np32(dy))
    assert rel_err(to_np32(dW), want, S) <= TOL[BF]
    dW2 = _run(lib, psi, xd, dyd, B, Cin, Cout)
    torch.cuda.synchronize()
    assert torch.equal(dW, dW2)  # fixed split order: bit-identical reruns


def test_weight_grad_full_size_sampled_channels(lib):
    """721x1440 -> 361x720, B=1, C=256, K=9: every dW[o, c, k] for a few input
    channels c (the oracle recomputes the forward only for those channels)."""
    w = WORKLOADS["down_fused_bwd_721x1440_to_361x720"]
    inp = make_inputs(w)
    ref = oracle.build_psi(w.grid_in, w.grid_out, w.kind, w.nrad, w.cutoff)
    psi = lib.Psi(w.grid_in, w.grid_out, w.kind, w.nrad, w.cutoff)
    dW = _run(lib, psi, inp["x"].cuda(), inp["dy"].cuda(), w.B, w.C, w.Cout)
    torch.cuda.synchronize()
    assert lib.disco_device_status() == 0
    chans = [0, 1, 127, w.C - 1]
    xs = inp["x"][:, chans].float().numpy()
    X, SX = oracle.fwd(ref, xs)
    want, S = oracle.einsum_w(inp["dy"].float().numpy(), X, SX)
    got = dW[:, chans].float().cpu().numpy()
    assert rel_err(got, want, S) <= TOL[BF]


def test_weight_grad_rejects_unsupported(lib):
    psi36 = lib.Psi((16, 36, 0), (16, 36, 0), 0, 3, 2 * math.pi / 16)  # W_in % 8 != 0
    assert lib.disco_fused_conv_bwd_weight_workspace_bytes(psi36.c, 1, 16, 16) == 0
    x = torch.zeros((1, 16, 16, 36), dtype=BF, device="cuda")
    dy = torch.zeros((1, 16, 16, 36), dtype=BF, device="cuda")
    dW = torch.zeros((16, 16, 3), dtype=BF, device="cuda")
    ws = torch.empty(256, dtype=torch.uint8, device="cuda")
    with pytest.raises(lib.DiscoError) as e:
        lib.disco_fused_conv_bwd_weight(psi36.c, x, dy, dW, 1, 16, 16, ws)
    assert e.value.status == -2
    psi = lib.Psi((16, 64, 0), (16, 64, 0), 0, 3, 2 * math.pi / 16)
    n = lib.disco_fused_conv_bwd_weight_workspace_bytes(psi.c, 1, 32, 16)
    assert n > 0
    x = torch.zeros((1, 32, 16, 64), dtype=BF, device="cuda")
    dy = torch.zeros((1, 16, 16, 64), dtype=BF, device="cuda")
    dW = torch.zeros((16, 32, 3), dtype=BF, device="cuda")
    small = torch.empty(256, dtype=torch.uint8, device="cuda")
    with pytest.raises(lib.DiscoError) as e:
        lib.disco_fused_conv_bwd_weight(psi.c, x, dy, dW, 1, 32, 16, small)  # workspace too small
    assert e.value.status == -7
