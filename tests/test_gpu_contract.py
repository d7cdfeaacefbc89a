"""disco_fwd / disco_bwd against the fp64 oracle, element by element on
small cases (several tiles and ragged tails) and on sampled outputs at the
full workload sizes, with NaN canaries and a determinism check."""
import math

import numpy as np
import pytest
import torch

import oracle
from sparse_spherical_convolution_gb300.workloads import PAGE_WORKLOADS, WORKLOADS, make_inputs, sample_points
from tests._helpers import TOL, rel_err, to_np32

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    from sparse_spherical_convolution_gb300 import build
    build.build()
    import sparse_spherical_convolution_gb300 as d
    return d


# (grid_in, grid_out, kind, nrad, cutoff, B, C, dtype)
SMALL = [
    ((16, 32, 0), (16, 32, 0), 0, 3, 2 * math.pi / 16, 1, 2, torch.float32),
    ((16, 32, 0), (16, 32, 0), 0, 3, 2 * math.pi / 16, 3, 5, torch.bfloat16),   # ragged channels
    ((64, 128, 0), (64, 128, 0), 0, 5, 3 * math.pi / 64, 2, 19, torch.bfloat16),
    ((128, 256, 0), (64, 128, 0), 1, 3, 3 * math.pi / 64, 1, 33, torch.bfloat16),
    ((128, 256, 0), (64, 128, 0), 1, 3, 3 * math.pi / 64, 1, 7, torch.float32),
    ((9, 16, 1), (9, 16, 1), 1, 3, 2 * math.pi / 8, 2, 3, torch.float32),        # full rings, empty ring
    ((17, 32, 1), (9, 16, 1), 1, 2, 3 * math.pi / 8, 1, 40, torch.bfloat16),     # s = 2, poles
    ((10, 24, 0), (10, 12, 0), 0, 1, 0.9, 2, 3, torch.bfloat16),                  # scalar stores
    ((37, 200, 1), (37, 200, 1), 1, 3, 4 * math.pi / 36, 1, 35, torch.bfloat16),  # 4 tiles, ragged
    ((16, 31, 0), (16, 31, 0), 0, 2, 2 * math.pi / 16, 1, 3, torch.float32),      # odd width
    ((16, 32, 2), (16, 32, 2), 1, 3, 3 * math.pi / 16, 1, 5, torch.float32),      # Legendre-Gauss
    ((40, 128, 2), (40, 64, 2), 1, 3, 3 * math.pi / 40, 2, 70, torch.bfloat16),   # Legendre-Gauss, s = 2, tensor cores
    ((65, 256, 1), (32, 128, 2), 1, 3, 3 * math.pi / 32, 1, 130, torch.bfloat16), # poles -> Legendre-Gauss
    ((24, 72, 0), (12, 36, 0), 1, 3, 3 * math.pi / 12, 2, 20, torch.bfloat16),    # W_out % 8 != 0: non-persistent forward tiles
    ((24, 72, 0), (12, 36, 0), 1, 3, 3 * math.pi / 12, 1, 9, torch.float16),      # the same in fp16
    ((2, 8, 0), (2, 8, 0), 0, 1, 2.5, 1, 3, torch.float32),                        # 2 rows, cutoff near the whole sphere
    ((3, 16, 1), (3, 16, 1), 1, 2, 2.0, 1, 4, torch.bfloat16),                    # 3-row pole grid (zero-weight poles)
    ((2, 8, 2), (2, 8, 2), 1, 1, 2.5, 2, 2, torch.float32),                        # 2-row Legendre-Gauss grid
]


def _inputs(B, C, K, gi, go, dtype, seed):
    g = torch.Generator().manual_seed(seed)
    x = torch.randn((B, C, gi[0], gi[1]), generator=g).to(dtype)
    G = torch.randn((B, C, K, go[0], go[1]), generator=g).to(dtype)
    return x, G


@pytest.mark.parametrize("case", SMALL, ids=lambda c: f"{c[0]}->{c[1]}-B{c[5]}C{c[6]}-{str(c[7])[6:]}")
def test_fwd_bwd_full_compare(lib, case):
    gi, go, kind, nrad, cut, B, C, dt = case
    ref = oracle.build_psi(gi, go, kind, nrad, cut)
    psi = lib.Psi(gi, go, kind, nrad, cut)
    x, G = _inputs(B, C, ref.K, gi, go, dt, 7)
    xd, Gd = x.cuda(), G.cuda()
    X = torch.full((B, C, ref.K, go[0], go[1]), float("nan"), dtype=dt, device="cuda")
    gx = torch.full((B, C, gi[0], gi[1]), float("nan"), dtype=dt, device="cuda")
    lib.disco_fwd(psi.c, xd, X, B, C)
    lib.disco_bwd(psi.c, Gd, gx, B, C)
    torch.cuda.synchronize()
    assert not torch.isnan(X).any() and not torch.isnan(gx).any()
    Xo, SX = oracle.fwd(ref, to_np32(x))
    go_, Sg = oracle.bwd(ref, to_np32(G))
    assert rel_err(to_np32(X), Xo, SX) <= TOL[dt]
    assert rel_err(to_np32(gx), go_, Sg) <= TOL[dt]
    # deterministic: no atomics, same result bit for bit
    X2 = torch.empty_like(X)
    gx2 = torch.empty_like(gx)
    lib.disco_fwd(psi.c, xd, X2, B, C)
    lib.disco_bwd(psi.c, Gd, gx2, B, C)
    torch.cuda.synchronize()
    assert torch.equal(X, X2) and torch.equal(gx, gx2)


@pytest.mark.parametrize("name", [n for n in WORKLOADS if WORKLOADS[n].grid_in[0] <= 128])
def test_workload_fwd_bwd_full(lib, name):
    """Every output of the small workloads (the contraction shapes)."""
    w = WORKLOADS[name]
    inp = make_inputs(w, with_G=True)
    ref = oracle.build_psi(w.grid_in, w.grid_out, w.kind, w.nrad, w.cutoff)
    psi = lib.Psi(w.grid_in, w.grid_out, w.kind, w.nrad, w.cutoff)
    B, C = w.B, w.C
    X = torch.empty(w.shapes()["X"], dtype=w.torch_dtype, device="cuda")
    gx = torch.empty(w.shapes()["x"], dtype=w.torch_dtype, device="cuda")
    lib.disco_fwd(psi.c, inp["x"].cuda(), X, B, C)
    lib.disco_bwd(psi.c, inp["G"].cuda(), gx, B, C)
    torch.cuda.synchronize()
    if w.B * w.C <= 128:
        Xo, SX = oracle.fwd(ref, to_np32(inp["x"]))
        go_, Sg = oracle.bwd(ref, to_np32(inp["G"]))
        assert rel_err(to_np32(X), Xo, SX) <= TOL[w.torch_dtype]
        assert rel_err(to_np32(gx), go_, Sg) <= TOL[w.torch_dtype]
    else:
        _sampled_check(ref, w, inp, X, gx, 4000)


def _sampled_check(ref, w, inp, X, gx, n):
    BC = w.B * w.C
    Xs = X.view(BC, w.K, w.grid_out[0], w.grid_out[1])
    p4 = sample_points((BC, w.K, w.grid_out[0], w.grid_out[1]), n, w.seed)
    v, S = oracle.fwd_points(ref, inp["x"].float().numpy(), p4.numpy())
    got = Xs[tuple(p4.cuda().T)].float().cpu().numpy()
    assert rel_err(got, v, S) <= TOL[w.torch_dtype]
    gs = gx.view(BC, w.grid_in[0], w.grid_in[1])
    p3 = sample_points((BC, w.grid_in[0], w.grid_in[1]), n, w.seed + 1)
    v, S = oracle.bwd_points(ref, inp["G"].float().numpy(), p3.numpy())
    got = gs[tuple(p3.cuda().T)].float().cpu().numpy()
    assert rel_err(got, v, S) <= TOL[w.torch_dtype]


FULL = {**{n: w for n, w in WORKLOADS.items() if w.grid_in[0] > 128}, **PAGE_WORKLOADS}


@pytest.mark.parametrize("name", list(FULL))
def test_workload_fwd_bwd_sampled_full_size(lib, name):
    """Full-size workloads (the benchmark's, in its launch configuration, and
    the page's Legendre-Gauss shapes), checked on sampled outputs (polar rows
    and the first/last elements included)."""
    w = FULL[name]
    ref = oracle.build_psi(w.grid_in, w.grid_out, w.kind, w.nrad, w.cutoff)
    psi = lib.Psi(w.grid_in, w.grid_out, w.kind, w.nrad, w.cutoff)
    inp = make_inputs(w, with_G=True)
    X = torch.empty(w.shapes()["X"], dtype=w.torch_dtype, device="cuda")
    gx = torch.empty(w.shapes()["x"], dtype=w.torch_dtype, device="cuda")
    lib.disco_fwd(psi.c, inp["x"].cuda(), X, w.B, w.C)
    lib.disco_bwd(psi.c, inp["G"].cuda(), gx, w.B, w.C)
    torch.cuda.synchronize()
    assert not torch.isnan(X.view(-1)[:: 9973]).any()
    _sampled_check(ref, w, inp, X, gx, 3000)
    # polar and equatorial rows explicitly
    BC = w.B * w.C
    Ho = w.grid_out[0]
    pts = np.array([[b, k, ho, wo] for b in (0, BC - 1) for k in range(w.K)
                    for ho in (0, 1, Ho // 2, Ho - 2, Ho - 1) for wo in (0, 7, w.grid_out[1] - 1)])
    v, S = oracle.fwd_points(ref, inp["x"].float().numpy(), pts)
    Xs = X.view(BC, w.K, Ho, w.grid_out[1])
    got = Xs[tuple(torch.from_numpy(pts).cuda().T)].float().cpu().numpy()
    assert rel_err(got, v, S) <= TOL[w.torch_dtype]


def test_concurrent_streams_same_psi(lib):
    """Launches on two streams at once with one psi.  The persistent
    tensor-core kernels hand out tiles from a counter private to each launch,
    so every result equals the one computed alone, bit for bit."""
    gi, go = (181, 360, 1), (181, 360, 1)
    psi = lib.Psi(gi, go, 1, 3, 4 * math.pi / 180)
    B, C, K = 2, 128, psi.c.K
    g = torch.Generator(device="cuda").manual_seed(11)
    xs = [torch.randn((B, C, gi[0], gi[1]), generator=g, device="cuda").to(torch.bfloat16) for _ in range(3)]
    Gs = [torch.randn((B, C, K, go[0], go[1]), generator=g, device="cuda").to(torch.bfloat16) for _ in range(3)]
    alone_X, alone_gx = [], []
    for x, G in zip(xs, Gs):
        X = torch.empty((B, C, K, go[0], go[1]), dtype=torch.bfloat16, device="cuda")
        gx = torch.empty_like(x)
        lib.disco_fwd(psi.c, x, X, B, C)
        lib.disco_bwd(psi.c, G, gx, B, C)
        alone_X.append(X)
        alone_gx.append(gx)
    torch.cuda.synchronize()
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    outs = []
    for rep in range(2):
        for i, (x, G) in enumerate(zip(xs, Gs)):
            X = torch.full((B, C, K, go[0], go[1]), float("nan"), dtype=torch.bfloat16, device="cuda")
            gx = torch.full_like(x, float("nan"))
            torch.cuda.synchronize()
            sa, sb = (s1, s2) if (i + rep) % 2 == 0 else (s2, s1)
            lib.disco_bwd(psi.c, G, gx, B, C, stream=sa)
            lib.disco_fwd(psi.c, x, X, B, C, stream=sb)
            lib.disco_bwd(psi.c, G, gx, B, C, stream=sb)  # same output again, racing the first
            outs.append((i, X, gx))
    torch.cuda.synchronize()
    assert lib.disco_device_status(clear=True) == 0
    for i, X, gx in outs:
        assert torch.equal(X, alone_X[i]) and torch.equal(gx, alone_gx[i])
