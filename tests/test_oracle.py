"""Pins of the fp64 CPU oracle against facts other than itself.

* dense brute force with independent 3-D vector geometry (chord distance,
  tangent-plane bearing) evaluated at the true output longitude: pins the
  distance, bearing sign, quadrature, normalisation, support rule, the
  longitude shift and the CSR indexing;
* the adjoint identity <psi x, g> = <x, psi^T g>: pins the transpose;
* longitude equivariance (bitwise): pins the shift direction;
* the indicator basis (K=1, psi=1 on the neighbourhood) against a plain
  neighbourhood sum: pins the neighbourhood rule;
* hand-derived closed forms on a 2x4 grid (tests/golden/closed_form_2x4.txt);
* hat partition of unity, constant-field normalisation, psi symmetries;
* the einsum against numpy.einsum (a textbook contraction);
* the error scale S = sum |terms| of every output (the denominator of every
  parity bar) against |M| of the dense brute force and numpy.einsum of
  absolute values, with planted mistakes (S summed over k, |W| dropped).
"""
import math
import os

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")

# tiny cases: (grid_in, grid_out, kind, nrad, cutoff)
TINY = [
    ((8, 16, 0), (8, 16, 0), oracle.ISO, 3, 2 * math.pi / 8),
    ((16, 32, 0), (16, 32, 0), oracle.ISO, 3, 2 * math.pi / 16),
    ((16, 32, 0), (8, 16, 0), oracle.ANISO, 3, 3 * math.pi / 8),
    ((9, 16, 1), (9, 16, 1), oracle.ANISO, 3, 2 * math.pi / 8),
    ((17, 32, 1), (9, 16, 1), oracle.ANISO, 2, 3 * math.pi / 8),
    ((12, 24, 0), (12, 24, 0), oracle.ANISO, 3, 4 * math.pi / 12),
    ((8, 16, 0), (8, 8, 0), oracle.ISO, 2, 3 * math.pi / 8),   # s = 2 with equal rows
    ((8, 16, 2), (8, 16, 2), oracle.ISO, 3, 2 * math.pi / 8),   # Legendre-Gauss grids
    ((16, 32, 0), (8, 16, 2), oracle.ANISO, 3, 3 * math.pi / 8),  # equiangular -> Legendre-Gauss, s = 2
]


def _colats(nlat, poles):
    if poles == 2:
        # numpy's Gauss-Legendre rule (ascending nodes): colatitudes north to south
        x, w = np.polynomial.legendre.leggauss(nlat)
        return np.arccos(x[::-1]), w[::-1].copy()
    if poles:
        th = np.arange(nlat) * math.pi / (nlat - 1)
        th[-1] = math.pi
        q = np.sin(th)
        q[0] = q[-1] = 0.0
    else:
        th = (np.arange(nlat) + 0.5) * math.pi / nlat
        q = np.sin(th)
    return th, q


def _unit(th, ph):
    th, ph = np.broadcast_arrays(np.asarray(th, float), np.asarray(ph, float))
    return np.stack([np.sin(th) * np.cos(ph), np.sin(th) * np.sin(ph), np.cos(th)], -1)


def _vector_dense(gi, go, kind, nrad, cutoff):
    """Independent dense matrix: chord-length distance and tangent-plane bearing."""
    Hin, Win, pin = gi
    Hout, Wout, pout = go
    thi, qi = _colats(Hin, pin)
    tho, _ = _colats(Hout, pout)
    phi_i = 2 * math.pi * np.arange(Win) / Win
    phi_o = 2 * math.pi * np.arange(Wout) / Wout
    Pi = _unit(thi[:, None], phi_i[None, :]).reshape(-1, 3)          # [Hin*Win, 3]
    Q = np.repeat(qi, Win)
    K = nrad if kind == oracle.ISO else 3 * nrad
    width = cutoff / nrad
    M = np.zeros((K, Hout, Wout, Hin * Win))
    for ho in range(Hout):
        for wo in range(Wout):
            t, p = tho[ho], phi_o[wo]
            po = _unit(t, p)
            north = np.array([-math.cos(t) * math.cos(p), -math.cos(t) * math.sin(p), math.sin(t)])
            east = np.array([-math.sin(p), math.cos(p), 0.0])
            chord = np.linalg.norm(Pi - po, axis=1)
            d = 2 * np.arcsin(np.clip(chord / 2, 0, 1))
            v = Pi - (Pi @ po)[:, None] * po
            beta = np.arctan2(v @ east, v @ north)
            for r in range(nrad):
                h = np.maximum(0.0, 1 - np.abs(d - r * width) / width)
                st = (h > 1e-9) & (Q > 0)
                N = np.sum(np.where(st, h * Q, 0.0))
                base = np.where(st, h * Q, 0.0) / N if N > 0 else np.zeros_like(h)
                if kind == oracle.ISO:
                    M[r, ho, wo] = base
                else:
                    far = d >= 1e-12
                    M[3 * r, ho, wo] = base
                    M[3 * r + 1, ho, wo] = np.where(far, base * np.cos(beta), 0.0)
                    M[3 * r + 2, ho, wo] = np.where(far, base * np.sin(beta), 0.0)
    return M.reshape(K * Hout * Wout, Hin * Win)


@pytest.mark.parametrize("case", TINY, ids=lambda c: f"{c[0]}->{c[1]}-k{c[2]}r{c[3]}")
def test_dense_bruteforce_vector_geometry(case):
    gi, go, kind, nrad, cut = case
    psi = oracle.build_psi(gi, go, kind, nrad, cut)
    M = _vector_dense(gi, go, kind, nrad, cut)
    rng = np.random.default_rng(0)
    x = rng.standard_normal((2, 1, gi[0], gi[1]))
    X, S = oracle.fwd(psi, x)
    ref = (M @ x.reshape(2, -1).T).T.reshape(X.shape)
    scale = np.abs(M) @ np.abs(x.reshape(2, -1).T)
    err = np.abs(X - ref) / np.maximum(scale.T.reshape(X.shape), 1e-300)
    assert err.max() < 1e-12
    # the C dense matrix (unshifted, per-row normalisation) agrees too
    Mc = oracle.dense_matrix(gi, go, kind, nrad, cut)
    assert np.abs(Mc - M).max() < 1e-12


@pytest.mark.parametrize("case", TINY, ids=lambda c: f"{c[0]}->{c[1]}")
def test_adjoint_identity(case):
    gi, go, kind, nrad, cut = case
    psi = oracle.build_psi(gi, go, kind, nrad, cut)
    rng = np.random.default_rng(1)
    x = rng.standard_normal((2, 3, gi[0], gi[1]))
    g = rng.standard_normal((2, 3, psi.K, go[0], go[1]))
    X, _ = oracle.fwd(psi, x)
    gx, _ = oracle.bwd(psi, g)
    lhs, rhs = np.vdot(X, g), np.vdot(x, gx)
    assert abs(lhs - rhs) <= 1e-12 * (np.abs(X).ravel() @ np.abs(g).ravel())


def test_adjoint_identity_workload_shapes():
    """The adjoint identity on every workload's grids (batch and channels reduced)."""
    from sparse_spherical_convolution_gb300.workloads import WORKLOADS
    rng = np.random.default_rng(2)
    for w in WORKLOADS.values():
        psi = oracle.build_psi(w.grid_in, w.grid_out, w.kind, w.nrad, w.cutoff)
        x = rng.standard_normal((1, 1) + tuple(w.grid_in[:2]))
        g = rng.standard_normal((1, 1, psi.K) + tuple(w.grid_out[:2]))
        X, _ = oracle.fwd(psi, x)
        gx, _ = oracle.bwd(psi, g)
        assert abs(np.vdot(X, g) - np.vdot(x, gx)) <= 1e-12 * (np.abs(X).ravel() @ np.abs(g).ravel())


@pytest.mark.parametrize("case", TINY, ids=lambda c: f"{c[0]}->{c[1]}")
def test_longitude_equivariance_bitwise(case):
    gi, go, kind, nrad, cut = case
    psi = oracle.build_psi(gi, go, kind, nrad, cut)
    s = gi[1] // go[1]
    rng = np.random.default_rng(3)
    x = rng.standard_normal((1, 2, gi[0], gi[1]))
    X, _ = oracle.fwd(psi, x)
    Xr, _ = oracle.fwd(psi, np.roll(x, s, axis=-1))
    assert np.array_equal(Xr, np.roll(X, 1, axis=-1))


@pytest.mark.parametrize("gi,go,cut", [
    ((16, 32, 0), (16, 32, 0), 2 * math.pi / 16),
    ((16, 32, 0), (8, 16, 0), 3 * math.pi / 8),
    ((9, 16, 1), (9, 16, 1), 3 * math.pi / 8),
    ((12, 24, 0), (12, 24, 0), 3 * math.pi / 12),   # ties on the meridian at d = cutoff
])
def test_indicator_basis_is_neighbourhood_sum(gi, go, cut):
    psi = oracle.build_psi(gi, go, oracle.INDICATOR, 1, cut)
    rng = np.random.default_rng(4)
    x = rng.standard_normal((1, 1, gi[0], gi[1]))
    X, _ = oracle.fwd(psi, x)
    thi, _ = _colats(gi[0], gi[2])
    tho, _ = _colats(go[0], go[2])
    Pi = _unit(thi[:, None], 2 * math.pi * np.arange(gi[1])[None, :] / gi[1]).reshape(-1, 3)
    xf = x.reshape(-1)
    for ho in range(go[0]):
        for wo in range(go[1]):
            po = _unit(tho[ho], 2 * math.pi * wo / go[1])
            d = 2 * np.arcsin(np.clip(np.linalg.norm(Pi - po, axis=1) / 2, 0, 1))
            ref = xf[(1 - d / cut) > 1e-9].sum()
            assert abs(X[0, 0, 0, ho, wo] - ref) < 1e-12 * np.abs(xf).sum()


def test_closed_form_golden_2x4():
    h1 = 1 - math.pi / 3.6
    D = 1 + 2 * h1
    env = {"h1": h1, "D": D, "sqrt": math.sqrt}
    rows = []
    with open(os.path.join(GOLDEN, "closed_form_2x4.txt")) as f:
        for line in f:
            line = line.split("#")[0].strip()
            if line:
                kind, k, hi, wi, expr = line.split()
                rows.append((kind, int(k), int(hi), int(wi), eval(expr, {}, env)))
    assert len(rows) == 12
    for kindname, kind in (("iso", oracle.ISO), ("aniso", oracle.ANISO)):
        psi = oracle.build_psi((2, 4, 0), (2, 4, 0), kind, 1, 1.2)
        assert psi.row_ptr[1] == 3
        assert psi.idx[:3].tolist() == [[0, 3], [0, 0], [0, 1]]
        for kn, k, hi, wi, v in rows:
            if kn != kindname:
                continue
            e = [tuple(t) for t in psi.idx[:3].tolist()].index((hi, wi))
            assert abs(psi.val[e, k] - v) < 1e-15, (kn, k, hi, wi)


@pytest.mark.parametrize("n", [2, 3, 16, 64, 361])
def test_gauss_legendre_nodes_and_weights(n):
    """Legendre-Gauss grid: nodes and weights against numpy's Gauss-Legendre
    rule, the weight sum 2, exactness on polynomials of degree < 2n, and the
    grid's colatitudes (ascending, symmetric about the equator)."""
    xs, ws = np.polynomial.legendre.leggauss(n)
    got = np.array([oracle.gauss_node(n, i) for i in range(n)])
    assert np.all(np.diff(got[:, 0]) < 0)
    assert np.abs(got[::-1, 0] - xs).max() < 1e-14
    # absolute: numpy's own weights are off by a few 1e-15 for large n (the
    # exactness checks below pin ours more tightly)
    assert np.abs(got[::-1, 1] - ws).max() < 2e-14
    assert abs(got[:, 1].sum() - 2.0) < 1e-13
    for deg in (0, 1, 2, 2 * n - 2, 2 * n - 1):
        exact = 0.0 if deg % 2 else 2.0 / (deg + 1)
        assert abs(np.sum(got[:, 1] * got[:, 0] ** deg) - exact) < 1e-12
    th = np.array([oracle.colat(n, 2, i) for i in range(n)])
    q = np.array([oracle.quad(n, 2, i) for i in range(n)])
    assert np.all(np.diff(th) > 0) and th[0] > 0 and th[-1] < math.pi
    assert np.abs(th + th[::-1] - math.pi).max() < 1e-13
    assert np.array_equal(q, got[:, 1])


def test_hat_partition_of_unity_and_nodes():
    width = 0.1
    for R in (2, 3, 5):
        for d in np.linspace(0, (R - 1) * width, 37):
            assert abs(sum(oracle.hat(d, r, width) for r in range(R)) - 1) < 1e-14
        for r in range(R):
            assert oracle.hat(r * width, r, width) == 1.0
            assert oracle.hat((r + 1) * width, r, width) < 1e-15
    assert oracle.hat(3.0 * width, 2, width) < 1e-15   # last hat vanishes at the cutoff


def test_geometry_textbook_cases():
    # along a meridian the distance is the colatitude difference, bearing north/south
    d, b = oracle.geometry(1.0, 0.7, 0, 64)
    assert abs(d - 0.3) < 1e-15 and abs(b) < 1e-15
    d, b = oracle.geometry(1.0, 1.3, 0, 64)
    assert abs(d - 0.3) < 1e-15 and abs(abs(b) - math.pi) < 1e-15
    # on the equator the distance is the longitude difference, bearing east/west
    d, b = oracle.geometry(math.pi / 2, math.pi / 2, 4, 64)
    assert abs(d - 2 * math.pi * 4 / 64) < 1e-15 and abs(b - math.pi / 2) < 1e-15
    d, b = oracle.geometry(math.pi / 2, math.pi / 2, -4, 64)
    assert abs(b + math.pi / 2) < 1e-15
    # antipodes
    d, _ = oracle.geometry(0.25, math.pi - 0.25, 32, 64)
    assert abs(d - math.pi) < 1e-12


@pytest.mark.parametrize("case", TINY, ids=lambda c: f"{c[0]}->{c[1]}")
def test_constant_field_and_symmetries(case):
    gi, go, kind, nrad, cut = case
    psi = oracle.build_psi(gi, go, kind, nrad, cut)
    X, _ = oracle.fwd(psi, np.ones((1, 1, gi[0], gi[1])))
    X = X[0, 0]
    for k in range(psi.K):
        a = 0 if kind == oracle.ISO else k % 3
        rows = X[k]
        if a == 0:
            # 1 wherever ring r has support; a ring with no support (only
            # possible next to a zero-weight pole row) gives exactly 0
            assert ((np.abs(rows - 1) < 1e-13) | (rows == 0)).all()
            if go[2] != 1:
                assert np.abs(rows - 1).max() < 1e-13
        elif a == 2:
            assert np.abs(rows).max() < 1e-13
    # psi(delta) = psi(-delta) for a in {0, 1}; psi(-delta) = -psi(delta) for a = 2
    W = gi[1]
    for ho in range(go[0]):
        lo, hi_ = psi.row_ptr[ho], psi.row_ptr[ho + 1]
        ent = {(int(h), int(w)): psi.val[e] for e, (h, w) in zip(range(lo, hi_), psi.idx[lo:hi_])}
        for (h, w), v in ent.items():
            if (-w) % W == w:
                continue  # offset 0 and the antipodal column are their own mirror
            m = ent.get((h, (-w) % W))
            if m is None:
                # a full ring of even width holds the antipodal column once only
                assert len([1 for (hh, _) in ent if hh == h]) == W
                continue
            for k in range(psi.K):
                a = 0 if kind == oracle.ISO else k % 3
                if a == 2:
                    assert m[k] == -v[k]
                else:
                    assert m[k] == v[k]


@pytest.mark.parametrize("case", TINY, ids=lambda c: f"{c[0]}->{c[1]}")
def test_index_structure(case):
    """Neighbour order: hi ascending then signed offset ascending; each (ho, hi)
    segment is one contiguous wrapped window symmetric about offset 0."""
    gi, go, kind, nrad, cut = case
    psi = oracle.build_psi(gi, go, kind, nrad, cut)
    W = gi[1]
    for ho in range(go[0]):
        seg = psi.idx[psi.row_ptr[ho]:psi.row_ptr[ho + 1]]
        dl = ((seg[:, 1] + W // 2) % W) - W // 2
        key = seg[:, 0].astype(np.int64) * 4 * W + dl
        assert np.all(np.diff(key) > 0)
        for h in np.unique(seg[:, 0]):
            d = np.sort(dl[seg[:, 0] == h])
            assert np.all(np.diff(d) == 1)
            assert d[0] == -d[-1] or (len(d) == W)
    # CSR rows are the union entries whose ring is structural, in the same order
    for k in range(psi.K):
        for ho in range(go[0]):
            cols = psi.csr_col[psi.csr_row_ptr[k * go[0] + ho]:psi.csr_row_ptr[k * go[0] + ho + 1]]
            seg = psi.idx[psi.row_ptr[ho]:psi.row_ptr[ho + 1]]
            union_cols = seg[:, 0].astype(np.int64) * W + seg[:, 1]
            idx = [int(np.where(union_cols == c)[0][0]) for c in cols]
            assert idx == sorted(idx)


def test_einsum_against_numpy():
    rng = np.random.default_rng(5)
    W = rng.standard_normal((6, 4, 9))
    X = rng.standard_normal((2, 4, 9, 3, 5))
    y, Sy = oracle.einsum(W, X)
    ref = np.einsum("ock,bckhw->bohw", W, X)
    assert np.abs(y - ref).max() < 1e-12
    assert np.abs(Sy - np.einsum("ock,bckhw->bohw", np.abs(W), np.abs(X))).max() < 1e-12
    dy = rng.standard_normal((2, 6, 3, 5))
    dX, _ = oracle.einsum_t(W, dy)
    assert np.abs(dX - np.einsum("ock,bohw->bckhw", W, dy)).max() < 1e-12


def test_weight_gradient_against_numpy_and_adjoint():
    """dW of y = einsum(W, X): against numpy.einsum, and the adjoint identity
    <dW, V> = <dy, einsum(V, X)> with the (independently pinned) einsum."""
    rng = np.random.default_rng(15)
    B, Cin, K, Cout = 2, 4, 9, 6
    X = rng.standard_normal((B, Cin, K, 3, 5))
    dy = rng.standard_normal((B, Cout, 3, 5))
    dW, SdW = oracle.einsum_w(dy, X)
    assert np.abs(dW - np.einsum("bohw,bckhw->ock", dy, X)).max() < 1e-12
    assert np.abs(SdW - np.einsum("bohw,bckhw->ock", np.abs(dy), np.abs(X))).max() < 1e-12
    V = rng.standard_normal((Cout, Cin, K))
    y, _ = oracle.einsum(V, X)
    lhs, rhs = float(np.sum(dW * V)), float(np.sum(dy * y))
    assert abs(lhs - rhs) <= 1e-12 * max(1.0, abs(rhs))
    # a transposed operand (c and k swapped in X) breaks the identity
    Xt = np.ascontiguousarray(X.reshape(B, K, Cin, 3, 5).transpose(0, 2, 1, 3, 4))
    dWt, _ = oracle.einsum_w(dy, Xt)
    assert abs(float(np.sum(dWt * V)) - rhs) > 1e-6 * max(1.0, abs(rhs))


@pytest.mark.parametrize("case", TINY[:2], ids=lambda c: f"{c[0]}->{c[1]}")
def test_fused_weight_gradient_is_the_derivative(case):
    """The fused forward is linear in W, so <dy, y(W + V)> - <dy, y(W)> equals
    <dW, V> exactly (up to rounding), with dW from fused_bwd_weight."""
    gi, go, kind, nrad, cut = case
    psi = oracle.build_psi(gi, go, kind, nrad, cut)
    rng = np.random.default_rng(16)
    B, C, Cout = 2, 3, 4
    x = rng.standard_normal((B, C, gi[0], gi[1]))
    dy = rng.standard_normal((B, Cout, go[0], go[1]))
    W = rng.standard_normal((Cout, C, psi.K))
    V = rng.standard_normal((Cout, C, psi.K))
    dW, _ = oracle.fused_bwd_weight(psi, x, dy)
    y0, _ = oracle.fused(psi, x, W)
    y1, _ = oracle.fused(psi, x, W + V)
    lhs, rhs = float(np.sum(dy * (y1 - y0))), float(np.sum(dW * V))
    assert abs(lhs - rhs) <= 1e-10 * max(1.0, abs(rhs))


@pytest.mark.parametrize("case", TINY[:4], ids=lambda c: f"{c[0]}->{c[1]}")
def test_sampled_points_match_full_arrays(case):
    gi, go, kind, nrad, cut = case
    psi = oracle.build_psi(gi, go, kind, nrad, cut)
    rng = np.random.default_rng(6)
    B, C, Cout = 2, 3, 4
    x = rng.standard_normal((B, C, gi[0], gi[1])).astype(np.float32)
    G = rng.standard_normal((B, C, psi.K, go[0], go[1])).astype(np.float32)
    W = rng.standard_normal((Cout, C, psi.K)).astype(np.float32)
    dy = rng.standard_normal((B, Cout, go[0], go[1])).astype(np.float32)
    X, SX = oracle.fwd(psi, x)
    gx, Sg = oracle.bwd(psi, G)
    y, Sy = oracle.fused(psi, x, W)
    fgx, Sfg = oracle.fused_bwd_input(psi, dy, W)
    n = 50
    p4 = np.stack([rng.integers(0, B * C, n), rng.integers(0, psi.K, n),
                   rng.integers(0, go[0], n), rng.integers(0, go[1], n)], 1)
    v, s = oracle.fwd_points(psi, x, p4)
    Xf, SXf = X.reshape(B * C, psi.K, go[0], go[1]), SX.reshape(B * C, psi.K, go[0], go[1])
    ref = Xf[tuple(p4.T)]
    assert np.abs(v - ref).max() <= 1e-13 * SXf[tuple(p4.T)].max()
    p3 = np.stack([rng.integers(0, B * C, n), rng.integers(0, gi[0], n),
                   rng.integers(0, gi[1], n)], 1)
    v, s = oracle.bwd_points(psi, G, p3)
    gf = gx.reshape(B * C, gi[0], gi[1])
    assert np.abs(v - gf[tuple(p3.T)]).max() <= 1e-12 * max(1.0, s.max())
    assert np.abs(s - Sg.reshape(B * C, gi[0], gi[1])[tuple(p3.T)]).max() <= 1e-12 * max(1.0, s.max())
    py = np.stack([rng.integers(0, B, n), rng.integers(0, Cout, n),
                   rng.integers(0, go[0], n), rng.integers(0, go[1], n)], 1)
    v, s = oracle.fused_points(psi, x, W, py)
    assert np.abs(v - y[tuple(py.T)]).max() <= 1e-12 * s.max()
    assert np.abs(s - Sy[tuple(py.T)]).max() <= 1e-12 * s.max()
    pg = np.stack([rng.integers(0, B, n), rng.integers(0, C, n),
                   rng.integers(0, gi[0], n), rng.integers(0, gi[1], n)], 1)
    v, s = oracle.fused_bwd_points(psi, dy, W, pg)
    assert np.abs(v - fgx[tuple(pg.T)]).max() <= 1e-12 * max(1.0, s.max())
    assert np.abs(s - Sfg[tuple(pg.T)]).max() <= 1e-12 * max(1.0, s.max())


def test_planted_mistakes_are_caught():
    """A wrong shift direction or a transposed operand must fail the pins."""
    gi, go, kind, nrad, cut = TINY[2]
    psi = oracle.build_psi(gi, go, kind, nrad, cut)
    M = _vector_dense(gi, go, kind, nrad, cut)
    rng = np.random.default_rng(7)
    x = rng.standard_normal((1, 1, gi[0], gi[1]))
    X, _ = oracle.fwd(psi, x)
    ref = (M @ x.reshape(1, -1).T).T.reshape(X.shape)
    # mirrored input (a sign error in the longitude offset) changes the result
    Xm, _ = oracle.fwd(psi, x[..., ::-1])
    assert np.abs(Xm - ref).max() > 1e-3
    # a dropped sin component (bearing sign flip) is caught by the brute force
    bad = np.array(X)
    bad[:, :, 2::3] *= -1
    assert np.abs(bad - ref).max() > 1e-3


# ------------------------------------------------------------------ error scale
#
# Every parity bar divides by S = sum over the elementary terms of |term|.  The
# oracle returns S beside each output; these tests recompute it from the
# independent vector-geometry dense matrix M (|psi| is |M| entry by entry) and
# from numpy.einsum, so that an S inflated or deflated anywhere (summed over k,
# a dropped |W| factor, the wrong transpose) fails here.

def _rel(a, b):
    return float(np.max(np.abs(a - b) / np.maximum(np.abs(b), 1e-300)))


@pytest.mark.parametrize("case", TINY, ids=lambda c: f"{c[0]}->{c[1]}-k{c[2]}r{c[3]}")
def test_error_scale_of_the_contractions(case):
    gi, go, kind, nrad, cut = case
    psi = oracle.build_psi(gi, go, kind, nrad, cut)
    Ma = np.abs(_vector_dense(gi, go, kind, nrad, cut))     # [K*Hout*Wout, Hin*Win]
    rng = np.random.default_rng(8)
    B, C = 2, 2
    x = rng.standard_normal((B, C, gi[0], gi[1]))
    G = rng.standard_normal((B, C, psi.K, go[0], go[1]))
    _, SX = oracle.fwd(psi, x)
    ref = (Ma @ np.abs(x).reshape(B * C, -1).T).T.reshape(SX.shape)
    assert _rel(SX, ref) < 1e-12
    _, Sg = oracle.bwd(psi, G)
    ref = (Ma.T @ np.abs(G).reshape(B * C, -1).T).T.reshape(Sg.shape)
    assert _rel(Sg, ref) < 1e-12


@pytest.mark.parametrize("case", TINY[:5], ids=lambda c: f"{c[0]}->{c[1]}")
def test_error_scale_of_the_einsums_and_fused_paths(case):
    gi, go, kind, nrad, cut = case
    psi = oracle.build_psi(gi, go, kind, nrad, cut)
    K = psi.K
    Ma = np.abs(_vector_dense(gi, go, kind, nrad, cut))
    rng = np.random.default_rng(9)
    B, Cin, Cout = 2, 3, 4
    x = rng.standard_normal((B, Cin, gi[0], gi[1]))
    W = rng.standard_normal((Cout, Cin, K))
    dy = rng.standard_normal((B, Cout, go[0], go[1]))
    # einsum adjoint: SdX = sum_o |W[o,c,k]| |dy[b,o,p]|
    _, SdX = oracle.einsum_t(W, dy)
    ref_dX = np.einsum("ock,bohw->bckhw", np.abs(W), np.abs(dy))
    assert _rel(SdX, ref_dX) < 1e-12
    # fused forward: S = sum_{c,k} |W| sum_n |psi x| = einsum(|W|, |M| |x|)
    _, Sy = oracle.fused(psi, x, W)
    SX = (Ma @ np.abs(x).reshape(B * Cin, -1).T).T.reshape(B, Cin, K, go[0], go[1])
    ref_y = np.einsum("ock,bckhw->bohw", np.abs(W), SX)
    assert _rel(Sy, ref_y) < 1e-12
    # fused input gradient: S = |M|^T applied to sum_o |W| |dy|
    _, Sgx = oracle.fused_bwd_input(psi, dy, W)
    ref_gx = (Ma.T @ ref_dX.reshape(B * Cin, -1).T).T.reshape(Sgx.shape)
    assert _rel(Sgx, ref_gx) < 1e-12
    # weight gradient: S = sum_{b,p} |dy| (|M| |x|)
    _, SdW = oracle.fused_bwd_weight(psi, x, dy)
    ref_w = np.einsum("bohw,bckhw->ock", np.abs(dy), SX)
    assert _rel(SdW, ref_w) < 1e-12
    # the sampled-point forms return the same S at their points
    n = 40
    p4 = np.stack([rng.integers(0, B * Cin, n), rng.integers(0, K, n),
                   rng.integers(0, go[0], n), rng.integers(0, go[1], n)], 1)
    _, s = oracle.fwd_points(psi, x.astype(np.float32), p4)
    x32 = np.abs(x.astype(np.float32).astype(np.float64))
    SX32 = (Ma @ x32.reshape(B * Cin, -1).T).T.reshape(B * Cin, K, go[0], go[1])
    assert _rel(s, SX32[tuple(p4.T)]) < 1e-12
    py = np.stack([rng.integers(0, B, n), rng.integers(0, Cout, n),
                   rng.integers(0, go[0], n), rng.integers(0, go[1], n)], 1)
    _, s = oracle.fused_points(psi, x.astype(np.float32), W.astype(np.float32), py)
    W32 = np.abs(W.astype(np.float32).astype(np.float64))
    ref = np.einsum("ock,bckhw->bohw", W32, SX32.reshape(B, Cin, K, go[0], go[1]))
    assert _rel(s, ref[tuple(py.T)]) < 1e-12
    G = rng.standard_normal((B, Cin, K, go[0], go[1])).astype(np.float32)
    p3 = np.stack([rng.integers(0, B * Cin, n), rng.integers(0, gi[0], n), rng.integers(0, gi[1], n)], 1)
    _, s = oracle.bwd_points(psi, G, p3)
    ref = (Ma.T @ np.abs(G.astype(np.float64)).reshape(B * Cin, -1).T).T.reshape(B * Cin, gi[0], gi[1])
    assert _rel(s, ref[tuple(p3.T)]) < 1e-12
    pg = np.stack([rng.integers(0, B, n), rng.integers(0, Cin, n),
                   rng.integers(0, gi[0], n), rng.integers(0, gi[1], n)], 1)
    _, s = oracle.fused_bwd_points(psi, dy.astype(np.float32), W.astype(np.float32), pg)
    d32 = np.abs(dy.astype(np.float32).astype(np.float64))
    dX32 = np.einsum("ock,bohw->bckhw", W32, d32)
    ref = (Ma.T @ dX32.reshape(B * Cin, -1).T).T.reshape(B, Cin, gi[0], gi[1])
    assert _rel(s, ref[tuple(pg.T)]) < 1e-12


def test_error_scale_planted_mistakes_are_caught():
    """An S off by a factor (summed over k, or with |W| dropped) fails the pins."""
    gi, go, kind, nrad, cut = TINY[2]
    psi = oracle.build_psi(gi, go, kind, nrad, cut)
    Ma = np.abs(_vector_dense(gi, go, kind, nrad, cut))
    rng = np.random.default_rng(10)
    x = rng.standard_normal((1, 2, gi[0], gi[1]))
    _, SX = oracle.fwd(psi, x)
    ref = (Ma @ np.abs(x).reshape(2, -1).T).T.reshape(SX.shape)
    summed_over_k = np.repeat(SX.sum(axis=2, keepdims=True), psi.K, axis=2)
    assert _rel(summed_over_k, ref) > 1e-3
    assert _rel(SX * psi.K, ref) > 1e-3
    W = rng.standard_normal((3, 2, psi.K))
    dy = rng.standard_normal((1, 3, go[0], go[1]))
    _, SdX = oracle.einsum_t(W, dy)
    no_w = np.einsum("ock,bohw->bckhw", np.ones_like(W), np.abs(dy))
    assert _rel(no_w, np.einsum("ock,bohw->bckhw", np.abs(W), np.abs(dy))) > 1e-3
    assert _rel(SdX, np.einsum("ock,bohw->bckhw", np.abs(W), np.abs(dy))) < 1e-12
