"""disco_fused_conv and disco_fused_conv_bwd_input against the fp64 oracle:
element by element on small cases (ragged channel, column and M tiles), on
every output of the downsampling workload, and on sampled outputs of the
full-size workloads in the benchmark's launch configuration."""
import math

import numpy as np
import pytest
import torch

import oracle
from sparse_spherical_convolution_gb300.workloads import PAGE_WORKLOADS, WORKLOADS, make_inputs, sample_points
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
    ((16, 32, 0), (16, 32, 0), 0, 3, 2 * math.pi / 16, 1, 16, 16),
    ((32, 64, 0), (16, 32, 0), 1, 3, 3 * math.pi / 16, 2, 32, 48),
    ((64, 128, 0), (64, 128, 0), 0, 5, 3 * math.pi / 64, 2, 16, 130),     # 2 M tiles, ragged
    ((17, 32, 1), (9, 16, 1), 1, 2, 3 * math.pi / 8, 1, 48, 256),         # poles, s = 2, K = 6
    ((37, 200, 1), (37, 200, 1), 1, 3, 4 * math.pi / 36, 1, 16, 64),      # ragged 64-column tiles
    ((10, 24, 0), (10, 12, 0), 0, 1, 0.9, 3, 16, 20),                      # K = 1, narrow ring
    ((16, 36, 0), (16, 36, 0), 1, 3, 2 * math.pi / 16, 1, 16, 40),        # W_in % 8 != 0: on-chip path
    ((32, 64, 0), (16, 32, 0), 1, 3, 3 * math.pi / 16, 1, 24, 8),         # Cin % 16 != 0 (workspace path)
    ((33, 64, 1), (33, 64, 1), 1, 3, 3 * math.pi / 32, 2, 64, 48),        # TMA GEMMs: ragged pixel tile, 3 dX n-tiles
    ((24, 72, 0), (12, 36, 0), 1, 3, 3 * math.pi / 12, 1, 32, 24),        # X from the non-persistent forward tiles
]


def _inputs(B, Cin, Cout, K, gi, go, seed):
    g = torch.Generator().manual_seed(seed)
    x = torch.randn((B, Cin, gi[0], gi[1]), generator=g).to(BF)
    W = (torch.randn((Cout, Cin, K), generator=g) / math.sqrt(Cin * K)).to(BF)
    dy = torch.randn((B, Cout, go[0], go[1]), generator=g).to(BF)
    return x, W, dy


def _run_fused(lib, psi, x, W, B, Cin, Cout, go):
    y = torch.full((B, Cout, go[0], go[1]), float("nan"), dtype=BF, device="cuda")
    nws = lib.disco_fused_conv_workspace_bytes(psi.c, B, Cin, Cout)
    ws = torch.empty(max(nws, 16), dtype=torch.uint8, device="cuda") if nws else None
    lib.disco_fused_conv(psi.c, x, W, y, B, Cin, Cout, ws)
    return y


def _run_fused_bwd(lib, psi, dy, W, B, Cin, Cout, gi):
    gx = torch.full((B, Cin, gi[0], gi[1]), float("nan"), dtype=BF, device="cuda")
    nws = lib.disco_fused_conv_bwd_input_workspace_bytes(psi.c, B, Cin)
    ws = torch.empty(nws, dtype=torch.uint8, device="cuda")
    lib.disco_fused_conv_bwd_input(psi.c, dy, W, gx, B, Cin, Cout, ws)
    return gx


@pytest.mark.parametrize("case", SMALL, ids=lambda c: f"{c[0]}->{c[1]}-B{c[5]}Ci{c[6]}Co{c[7]}")
def test_fused_full_compare(lib, case):
    gi, go, kind, nrad, cut, B, Cin, Cout = case
    ref = oracle.build_psi(gi, go, kind, nrad, cut)
    psi = lib.Psi(gi, go, kind, nrad, cut)
    x, W, dy = _inputs(B, Cin, Cout, ref.K, gi, go, 11)
    xd, Wd, dyd = x.cuda(), W.cuda(), dy.cuda()
    y = _run_fused(lib, psi, xd, Wd, B, Cin, Cout, go)
    gx = _run_fused_bwd(lib, psi, dyd, Wd, B, Cin, Cout, gi)
    torch.cuda.synchronize()
    assert lib.disco_device_status() == 0
    assert not torch.isnan(y).any() and not torch.isnan(gx).any()
    yo, Sy = oracle.fused(ref, to_np32(x), to_np32(W))
    assert rel_err(to_np32(y), yo, Sy) <= TOL[BF]
    go_, Sg = oracle.fused_bwd_input(ref, to_np32(dy), to_np32(W))
    assert rel_err(to_np32(gx), go_, Sg) <= TOL[BF]
    # deterministic
    y2 = _run_fused(lib, psi, xd, Wd, B, Cin, Cout, go)
    gx2 = _run_fused_bwd(lib, psi, dyd, Wd, B, Cin, Cout, gi)
    torch.cuda.synchronize()
    assert torch.equal(y, y2) and torch.equal(gx, gx2)


def test_fused_matches_unfused_path(lib):
    """fused == einsum of the materialised contraction (both on the GPU),
    the page's fused == unfused check, within the bf16 tolerance."""
    gi, go, kind, nrad, cut, B, Cin, Cout = SMALL[1]
    psi = lib.Psi(gi, go, kind, nrad, cut)
    ref = oracle.build_psi(gi, go, kind, nrad, cut)
    x, W, _ = _inputs(B, Cin, Cout, ref.K, gi, go, 12)
    xd, Wd = x.cuda(), W.cuda()
    y = _run_fused(lib, psi, xd, Wd, B, Cin, Cout, go)
    X = torch.empty((B, Cin, ref.K, go[0], go[1]), dtype=torch.float32, device="cuda")
    lib.disco_fwd(psi.c, xd.float(), X, B, Cin)
    torch.cuda.synchronize()
    # plain torch einsum as the unfused second stage (test-side reference only)
    y_unfused = torch.einsum("ock,bckhw->bohw", Wd.float(), X)
    _, Sy = oracle.fused(ref, to_np32(x), to_np32(W))
    assert rel_err(to_np32(y), y_unfused.cpu().numpy(), Sy) <= TOL[BF]


def test_fused_workload_full(lib):
    """Every output of the downsampling fused workload."""
    w = WORKLOADS["down_fused_128x256_to_64x128"]
    inp = make_inputs(w)
    ref = oracle.build_psi(w.grid_in, w.grid_out, w.kind, w.nrad, w.cutoff)
    psi = lib.Psi(w.grid_in, w.grid_out, w.kind, w.nrad, w.cutoff)
    y = _run_fused(lib, psi, inp["x"].cuda(), inp["W"].cuda(), w.B, w.C, w.Cout, w.grid_out)
    torch.cuda.synchronize()
    assert lib.disco_device_status() == 0
    yo, Sy = oracle.fused(ref, to_np32(inp["x"]), to_np32(inp["W"]))
    assert rel_err(to_np32(y), yo, Sy) <= TOL[BF]


@pytest.mark.parametrize("name", ["fused_bwd_361x720", "down_fused_bwd_721x1440_to_361x720",
                                  "page_self_256x360x720_gauss", "page_self_512x360x720_gauss",
                                  "page_down_80x721x1440_to_360x720_gauss"])
def test_fused_workload_sampled_full_size(lib, name):
    w = WORKLOADS[name] if name in WORKLOADS else PAGE_WORKLOADS[name]
    inp = make_inputs(w)
    ref = oracle.build_psi(w.grid_in, w.grid_out, w.kind, w.nrad, w.cutoff)
    psi = lib.Psi(w.grid_in, w.grid_out, w.kind, w.nrad, w.cutoff)
    xd, Wd, dyd = inp["x"].cuda(), inp["W"].cuda(), inp["dy"].cuda()
    y = _run_fused(lib, psi, xd, Wd, w.B, w.C, w.Cout, w.grid_out)
    gx = _run_fused_bwd(lib, psi, dyd, Wd, w.B, w.C, w.Cout, w.grid_in)
    torch.cuda.synchronize()
    assert lib.disco_device_status() == 0
    assert not torch.isnan(y).any() and not torch.isnan(gx).any()
    Ho, Wo = w.grid_out[:2]
    py = sample_points((w.B, w.Cout, Ho, Wo), 1500, w.seed)
    extra = torch.tensor([[0, o, ho, wo] for o in (0, w.Cout - 1) for ho in (0, 1, Ho // 2, Ho - 1)
                          for wo in (0, 63, 64, Wo - 1)])
    py = torch.cat([py, extra])
    v, S = oracle.fused_points(ref, inp["x"].float().numpy(), inp["W"].float().numpy(), py.numpy())
    got = y[tuple(py.cuda().T)].float().cpu().numpy()
    assert rel_err(got, v, S) <= TOL[BF]
    Hi, Wi = w.grid_in[:2]
    pg = sample_points((w.B, w.C, Hi, Wi), 1500, w.seed + 1)
    extra = torch.tensor([[0, c, hi, wi] for c in (0, w.C - 1) for hi in (0, 1, Hi // 2, Hi - 2, Hi - 1)
                          for wi in (0, 1, Wi - 1)])
    pg = torch.cat([pg, extra])
    v, S = oracle.fused_bwd_points(ref, inp["dy"].float().numpy(), inp["W"].float().numpy(), pg.numpy())
    got = gx[tuple(pg.cuda().T)].float().cpu().numpy()
    assert rel_err(got, v, S) <= TOL[BF]


def test_fused_rejects_unsupported(lib):
    gi, go = (16, 64, 0), (16, 64, 0)  # tensor-core path (W_in % 8 == 0, W_in >= 64)
    psi = lib.Psi(gi, go, 0, 3, 2 * math.pi / 16)
    x = torch.zeros((1, 8, 16, 64), dtype=BF, device="cuda")
    W = torch.zeros((8, 8, 3), dtype=BF, device="cuda")
    y = torch.zeros((1, 8, 16, 64), dtype=BF, device="cuda")
    with pytest.raises(lib.DiscoError) as e:
        lib.disco_fused_conv(psi.c, x, W, y, 1, 8, 8)  # no workspace for the tensor-core path
    assert e.value.status == -7
    with pytest.raises(lib.DiscoError) as e:
        lib.disco_fused_conv(psi.c, x.float(), W.float(), y.float(), 1, 8, 8)  # fp32
    assert e.value.status == -2
    psi36 = lib.Psi((16, 36, 0), (16, 36, 0), 0, 3, 2 * math.pi / 16)  # on-chip path
    x36 = torch.zeros((1, 8, 16, 36), dtype=BF, device="cuda")
    y36 = torch.zeros((1, 8, 16, 36), dtype=BF, device="cuda")
    assert lib.disco_fused_conv_workspace_bytes(psi36.c, 1, 8, 8) == 0
    with pytest.raises(lib.DiscoError) as e:
        lib.disco_fused_conv(psi36.c, x36, W, y36, 1, 8, 8)  # Cin % 16 != 0 on the on-chip path
    assert e.value.status == -2
    ws = torch.empty(16, dtype=torch.uint8, device="cuda")
    with pytest.raises(lib.DiscoError) as e:
        lib.disco_fused_conv_bwd_input(psi.c, y, W, x, 1, 8, 8, ws)  # workspace too small
    assert e.value.status == -7
