"""fp16 inputs (the page's third precision) against the fp64 oracle: the
contractions on the tensor-core and CUDA-core paths, the fused convolution,
its input and weight gradients, a sampled full-size case, determinism and
the fp16 shape rules of the fused paths."""
import math

import numpy as np
import pytest
import torch

import oracle
from sparse_spherical_convolution_gb300.workloads import WORKLOADS, sample_points
from tests._helpers import TOL, rel_err, to_np32

pytestmark = pytest.mark.gpu
H = torch.float16


@pytest.fixture(scope="module")
def lib():
    from sparse_spherical_convolution_gb300 import build
    build.build()
    import sparse_spherical_convolution_gb300 as d
    d.disco_device_status(clear=True)
    return d


# (grid_in, grid_out, kind, nrad, cutoff, B, C)
CONTRACT = [
    ((64, 128, 0), (64, 128, 0), 0, 5, 3 * math.pi / 64, 2, 19),       # tensor cores, s = 1
    ((128, 256, 0), (64, 128, 0), 1, 3, 3 * math.pi / 64, 1, 33),      # tensor cores, s = 2
    ((37, 200, 1), (37, 200, 1), 1, 3, 4 * math.pi / 36, 1, 35),       # ragged tiles, poles
    ((10, 24, 0), (10, 12, 0), 0, 1, 0.9, 2, 3),                        # CUDA-core path
    ((16, 32, 2), (16, 32, 2), 1, 3, 3 * math.pi / 16, 1, 5),          # Legendre-Gauss, CUDA cores
]


def _gen(shape, g, scale=1.0):
    return (torch.randn(shape, generator=g) * scale).to(H)


@pytest.mark.parametrize("case", CONTRACT, ids=lambda c: f"{c[0]}->{c[1]}-B{c[5]}C{c[6]}")
def test_fp16_contractions(lib, case):
    gi, go, kind, nrad, cut, B, C = case
    ref = oracle.build_psi(gi, go, kind, nrad, cut)
    psi = lib.Psi(gi, go, kind, nrad, cut)
    g = torch.Generator().manual_seed(31)
    x = _gen((B, C, gi[0], gi[1]), g)
    G = _gen((B, C, ref.K, go[0], go[1]), g)
    X = torch.full((B, C, ref.K, go[0], go[1]), float("nan"), dtype=H, device="cuda")
    gx = torch.full((B, C, gi[0], gi[1]), float("nan"), dtype=H, device="cuda")
    lib.disco_fwd(psi.c, x.cuda(), X, B, C)
    lib.disco_bwd(psi.c, G.cuda(), gx, B, C)
    torch.cuda.synchronize()
    assert lib.disco_device_status() == 0
    Xo, SX = oracle.fwd(ref, to_np32(x))
    go_, Sg = oracle.bwd(ref, to_np32(G))
    assert rel_err(to_np32(X), Xo, SX) <= TOL[H]
    assert rel_err(to_np32(gx), go_, Sg) <= TOL[H]
    X2 = torch.empty_like(X)
    lib.disco_fwd(psi.c, x.cuda(), X2, B, C)
    torch.cuda.synchronize()
    assert torch.equal(X, X2)


# (grid_in, grid_out, kind, nrad, cutoff, B, Cin, Cout)
# (fp16 fused paths need the tensor-core GEMM shapes: Cout >= 64 and a
# multiple of 8, Cin*K a multiple of 64, for the input gradient)
FUSED = [
    ((33, 64, 1), (33, 64, 1), 1, 3, 3 * math.pi / 32, 2, 64, 64),      # ragged pixel tile
    ((128, 256, 0), (64, 128, 0), 1, 3, 3 * math.pi / 64, 1, 64, 136),  # s = 2, 2 o tiles
]


@pytest.mark.parametrize("case", FUSED, ids=lambda c: f"{c[0]}->{c[1]}-B{c[5]}Ci{c[6]}Co{c[7]}")
def test_fp16_fused_and_gradients(lib, case):
    gi, go, kind, nrad, cut, B, Cin, Cout = case
    ref = oracle.build_psi(gi, go, kind, nrad, cut)
    psi = lib.Psi(gi, go, kind, nrad, cut)
    K = ref.K
    g = torch.Generator().manual_seed(32)
    x = _gen((B, Cin, gi[0], gi[1]), g)
    W = _gen((Cout, Cin, K), g, 1 / math.sqrt(Cin * K))
    dy = _gen((B, Cout, go[0], go[1]), g)
    xd, Wd, dyd = x.cuda(), W.cuda(), dy.cuda()
    y = torch.full((B, Cout, go[0], go[1]), float("nan"), dtype=H, device="cuda")
    ws = torch.empty(lib.disco_fused_conv_workspace_bytes(psi.c, B, Cin, Cout, lib.DISCO_F16), dtype=torch.uint8,
                     device="cuda")
    lib.disco_fused_conv(psi.c, xd, Wd, y, B, Cin, Cout, ws)
    gx = torch.full((B, Cin, gi[0], gi[1]), float("nan"), dtype=H, device="cuda")
    wsb = torch.empty(lib.disco_fused_conv_bwd_input_workspace_bytes(psi.c, B, Cin, lib.DISCO_F16),
                      dtype=torch.uint8, device="cuda")
    lib.disco_fused_conv_bwd_input(psi.c, dyd, Wd, gx, B, Cin, Cout, wsb)
    dW = torch.full((Cout, Cin, K), float("nan"), dtype=H, device="cuda")
    nw = lib.disco_fused_conv_bwd_weight_workspace_bytes(psi.c, B, Cin, Cout, lib.DISCO_F16)
    assert nw > 0
    wsw = torch.empty(nw, dtype=torch.uint8, device="cuda")
    lib.disco_fused_conv_bwd_weight(psi.c, xd, dyd, dW, B, Cin, Cout, wsw)
    torch.cuda.synchronize()
    assert lib.disco_device_status() == 0
    yo, Sy = oracle.fused(ref, to_np32(x), to_np32(W))
    assert rel_err(to_np32(y), yo, Sy) <= TOL[H]
    gxo, Sg = oracle.fused_bwd_input(ref, to_np32(dy), to_np32(W))
    assert rel_err(to_np32(gx), gxo, Sg) <= TOL[H]
    dWo, Sw = oracle.fused_bwd_weight(ref, to_np32(x), to_np32(dy))
    assert rel_err(to_np32(dW), dWo, Sw) <= TOL[H]


def test_fp16_full_size_sampled(lib):
    """361x720 (poles), B=2, C=128, K=9 in fp16 on the tensor-core path:
    sampled outputs of disco_fwd and disco_bwd, polar rows included."""
    w = WORKLOADS["fused_bwd_361x720"]
    ref = oracle.build_psi(w.grid_in, w.grid_out, w.kind, w.nrad, w.cutoff)
    psi = lib.Psi(w.grid_in, w.grid_out, w.kind, w.nrad, w.cutoff)
    g = torch.Generator().manual_seed(33)
    sh = w.shapes()
    x = _gen(sh["x"], g)
    G = _gen(sh["X"], g)
    X = torch.empty(sh["X"], dtype=H, device="cuda")
    gx = torch.empty(sh["x"], dtype=H, device="cuda")
    lib.disco_fwd(psi.c, x.cuda(), X, w.B, w.C)
    lib.disco_bwd(psi.c, G.cuda(), gx, w.B, w.C)
    torch.cuda.synchronize()
    assert lib.disco_device_status() == 0
    BC, Ho, Wo = w.B * w.C, w.grid_out[0], w.grid_out[1]
    p4 = sample_points((BC, w.K, Ho, Wo), 1500, 33)
    extra = torch.tensor([[b, k, ho, wo] for b in (0, BC - 1) for k in (0, w.K - 1)
                          for ho in (0, 1, Ho // 2, Ho - 1) for wo in (0, Wo - 1)])
    p4 = torch.cat([p4, extra])
    v, S = oracle.fwd_points(ref, x.float().numpy(), p4.numpy())
    got = X.view(BC, w.K, Ho, Wo)[tuple(p4.cuda().T)].float().cpu().numpy()
    assert rel_err(got, v, S) <= TOL[H]
    p3 = sample_points((BC, w.grid_in[0], w.grid_in[1]), 1500, 34)
    v, S = oracle.bwd_points(ref, G.float().numpy(), p3.numpy())
    got = gx.view(BC, w.grid_in[0], w.grid_in[1])[tuple(p3.cuda().T)].float().cpu().numpy()
    assert rel_err(got, v, S) <= TOL[H]


def test_fp16_fused_shape_rules(lib):
    """fp16 fused calls take the tensor-core shapes only; others are
    rejected before any launch."""
    psi36 = lib.Psi((16, 36, 0), (16, 36, 0), 0, 3, 2 * math.pi / 16)  # W_in % 8 != 0
    x = torch.zeros((1, 16, 16, 36), dtype=H, device="cuda")
    W = torch.zeros((16, 16, 3), dtype=H, device="cuda")
    y = torch.zeros((1, 16, 16, 36), dtype=H, device="cuda")
    assert lib.disco_fused_conv_workspace_bytes(psi36.c, 1, 16, 16, lib.DISCO_F16) == 0
    with pytest.raises(lib.DiscoError) as e:
        lib.disco_fused_conv(psi36.c, x, W, y, 1, 16, 16)
    assert e.value.status == -2
    ws = torch.empty(lib.disco_fused_conv_bwd_input_workspace_bytes(psi36.c, 1, 16, lib.DISCO_F16),
                     dtype=torch.uint8, device="cuda")
    with pytest.raises(lib.DiscoError) as e:
        lib.disco_fused_conv_bwd_input(psi36.c, y, W, x, 1, 16, 16, ws)
    assert e.value.status == -2
