"""psi built on the GPU against the oracle: index structures bit-exact,
values within 1 fp32 ulp of the fp64 oracle rounded to fp32."""
import math

import numpy as np
import pytest
import torch

import oracle
from sparse_spherical_convolution_gb300.workloads import PAGE_WORKLOADS, WORKLOADS
from tests._helpers import ulp_diff_f32

pytestmark = pytest.mark.gpu

CASES = [(w.grid_in, w.grid_out, w.kind, w.nrad, w.cutoff) for w in WORKLOADS.values()] + [
    ((9, 16, 1), (9, 16, 1), 1, 3, 2 * math.pi / 8),       # coarse pole grid, empty ring at the pole
    ((17, 32, 1), (9, 16, 1), 1, 2, 3 * math.pi / 8),      # s = 2, pole grids
    ((12, 24, 0), (12, 24, 0), 1, 3, 4 * math.pi / 12),    # ties at d = cutoff on the meridian
    ((10, 24, 0), (10, 12, 0), 0, 1, 0.9),                 # K = 1, W_out not a multiple of 8
    ((16, 31, 0), (16, 31, 0), 0, 2, 2 * math.pi / 16),    # odd ring width
    ((8, 16, 2), (8, 16, 2), 0, 3, 2 * math.pi / 8),       # Legendre-Gauss grids
    ((33, 64, 1), (16, 32, 2), 1, 3, 3 * math.pi / 16),    # pole grid -> Legendre-Gauss, s = 2
    ((3, 16, 1), (3, 16, 1), 1, 2, 2.0),                   # 3-row pole grid, one input-row group
    ((2, 8, 2), (2, 8, 2), 1, 1, 2.5),                     # 2-row Legendre-Gauss grid, full rings
] + [(w.grid_in, w.grid_out, w.kind, w.nrad, w.cutoff) for w in PAGE_WORKLOADS.values()]


@pytest.fixture(scope="module")
def lib():
    from sparse_spherical_convolution_gb300 import build
    build.build()
    import sparse_spherical_convolution_gb300 as d
    return d


@pytest.mark.parametrize("case", CASES, ids=lambda c: f"{c[0]}->{c[1]}-k{c[2]}r{c[3]}")
def test_psi_bit_exact(lib, case):
    gi, go, kind, nrad, cut = case
    ref = oracle.build_psi(gi, go, kind, nrad, cut)
    psi = lib.Psi(gi, go, kind, nrad, cut)
    torch.cuda.synchronize()
    c = psi.c
    assert c.K == ref.K and c.nnz == ref.row_ptr[-1] and c.nnz_csr == ref.csr_row_ptr[-1]
    assert np.array_equal(psi.tensor("row_ptr").cpu().numpy(), ref.row_ptr)
    assert np.array_equal(psi.tensor("idx").cpu().numpy(), ref.idx)
    assert np.array_equal(psi.tensor("csr_row_ptr").cpu().numpy(), ref.csr_row_ptr)
    assert np.array_equal(psi.tensor("csr_col").cpu().numpy(), ref.csr_col)
    val = psi.tensor("val").cpu().numpy()
    assert np.all(val[:, ref.K:] == 0)
    _close_f32(val[:, :ref.K], ref.val)
    _close_f32(psi.tensor("csr_val").cpu().numpy(), ref.csr_val)


def _close_f32(gpu, ref64):
    """Each value within 1 fp32 ulp of the fp64 oracle rounded to fp32, except
    numerical zeros: a sin(bearing) that is 0 in exact arithmetic comes out as
    +-1e-16-ish from either libm (e.g. sin(pi)), so values below 1e-9 of the
    largest one are compared with that absolute floor instead."""
    ref32 = ref64.astype(np.float32)
    floor = 1e-9 * np.abs(ref64).max()
    small = np.abs(ref64) < floor
    assert np.all(np.abs(gpu[small].astype(np.float64) - ref64[small]) <= floor)
    assert ulp_diff_f32(gpu[~small], ref32[~small]) <= 1


@pytest.mark.parametrize("case", CASES[:3] + CASES[5:], ids=lambda c: f"{c[0]}->{c[1]}")
def test_runs_are_consistent_with_union_layout(lib, case):
    """The kernel-side run table, transposed runs and pair weights describe
    exactly the union layout."""
    gi, go, kind, nrad, cut = case
    psi = lib.Psi(gi, go, kind, nrad, cut)
    torch.cuda.synchronize()
    c = psi.c
    W = gi[1]
    row_ptr = psi.tensor("row_ptr").cpu().numpy()
    idx = psi.tensor("idx").cpu().numpy()
    val = psi.tensor("val").cpu().numpy()
    runs = psi.tensor("runs").cpu().numpy()
    run_ptr = psi.tensor("run_ptr").cpu().numpy()
    hval = psi.tensor("hval").cpu().numpy()
    covered = 0
    for ho in range(go[0]):
        rs = runs[run_ptr[ho]:run_ptr[ho + 1]]
        assert np.all(rs[:, 0] == ho) and np.all(np.diff(rs[:, 1]) > 0)
        e = row_ptr[ho]
        for (rho, hi, D, hoff, e0, ln, npair, anti) in rs:
            assert e0 == e
            seg = idx[e0:e0 + ln]
            assert np.all(seg[:, 0] == hi)
            dl = ((seg[:, 1] + W // 2) % W) - W // 2
            zero = e0 + int(np.where(dl == 0)[0][0])
            for d in range(npair + 1):
                scale = 0.5 if d == 0 else 1.0
                assert np.array_equal(hval[hoff + d], val[zero + d] * scale)
            if anti:
                assert np.array_equal(hval[hoff + npair + 1], val[e0] * 0.5)
            assert D == npair + anti
            e += ln
        covered += e - row_ptr[ho]
        assert e == row_ptr[ho + 1]
    assert covered == c.nnz
    trun_ptr = psi.tensor("trun_ptr").cpu().numpy()
    truns = psi.tensor("truns").cpu().numpy()
    for hi in range(gi[0]):
        rs = runs[truns[trun_ptr[hi]:trun_ptr[hi + 1]]]
        assert np.all(rs[:, 1] == hi) and np.all(np.diff(rs[:, 0]) > 0)
    order = psi.tensor("row_order").cpu().numpy()
    assert sorted(order.tolist()) == list(range(go[0]))
    work = np.diff(row_ptr)[order]
    assert np.all(np.diff(work) <= 0)
    _check_tables(psi, runs, val, gi, go)


def _bf16_bits(v):
    return torch.from_numpy(np.ascontiguousarray(v, np.float32)).to(torch.bfloat16).view(torch.int16).numpy()


def _f16_bits(v):
    return torch.from_numpy(np.ascontiguousarray(v, np.float32)).to(torch.float16).view(torch.int16).numpy()


def _check_tables(psi, runs, val, gi, go):
    """Forward tables and the transpose tables by input-row group hold exactly
    the bf16-rounded union values at the documented positions, zeros elsewhere;
    their fp16 copies the fp16-rounded values at the same positions."""
    K, W, s = psi.c.K, gi[1], gi[1] // go[1]
    ftab, foff = psi.tensor("ftab").cpu().numpy(), psi.tensor("ftab_off").cpu().numpy()
    ftab_h = psi.tensor("ftab_h").cpu().numpy()
    assert foff[-1] == psi.c.nftab
    ext = {}
    for r, (ho, hi, D, hoff, e0, ln, npair, anti) in enumerate(runs):
        dlo = -(W // 2) if ln == W else -npair
        dhi = dlo + ln - 1
        vb = _bf16_bits(val[e0:e0 + ln, :K])            # [len, K], offsets dlo..dhi
        vh = _f16_bits(val[e0:e0 + ln, :K])
        ext[(int(ho), int(hi))] = (dlo, dhi, vb, vh)
        TL = (ln + 16 + 7) // 8 * 8
        for tab, v in ((ftab, vb), (ftab_h, vh)):
            want = np.zeros((K, TL), np.int16)
            want[:, 8:8 + ln] = v.T
            assert np.array_equal(tab[foff[r]:foff[r] + K * TL].reshape(K, TL), want)
    _check_group_tables(psi, ext, gi, go)


def _halfwidth(dlo, dhi, s):
    """max(EH, -EL) with EH = floor(dhi / s), EL = ceil((dlo - s + 1) / s)."""
    EH = dhi // s
    EL = -((-(dlo - s + 1)) // s)
    return max(EH, -EL)


def _check_group_tables(psi, ext, gi, go):
    Hin, W = gi[0], gi[1]
    s, K = W // go[1], psi.c.K
    if s > 2:
        assert psi.c.ngrp == 0
        return
    TQ = 32 // s
    CW = (63 + TQ + 7) // 8 * 8
    BLK = 8 * s * CW
    nz = (Hin + 7) // 8
    assert psi.c.ngrp == nz
    gptr = psi.tensor("grp_ptr").cpu().numpy()
    grp = psi.tensor("grp").cpu().numpy()
    gtab = psi.tensor("gtab").cpu().numpy()
    gtab_h = psi.tensor("gtab_h").cpu().numpy()
    assert gptr[0] == 0 and gptr[-1] == psi.c.ngrp_ent
    assert psi.c.grp_max == int(np.diff(gptr).max())
    off_next = 0
    for z in range(nz):
        rows = range(8 * z, min(Hin, 8 * z + 8))
        hos = sorted({ho for (ho, hi) in ext if hi in rows})
        ents = grp[gptr[z]:gptr[z + 1]]
        assert [int(e[0]) for e in ents] == hos
        for e in ents:
            ho, off = int(e[0]), int(e[1])
            MW, KB, nch = int(e[2]) & 0xFFFF, int(e[2]) >> 16, int(e[3]) & 0xFFFF
            E = max(_halfwidth(dlo, dhi, s) for (h2, hi), (dlo, dhi, _, _) in ext.items()
                    if h2 == ho and hi in rows)
            assert MW == (E + 7) // 8 * 8
            assert KB == (TQ + 2 * MW + 15) // 16 and nch == (KB + 3) // 4
            # the first and last row of the group with support at ho
            sup = [r for r, hi in enumerate(rows) if (ho, hi) in ext]
            assert ((int(e[3]) >> 16) & 0xFF, (int(e[3]) >> 24) & 0xFF) == (sup[0], sup[-1])
            assert off == off_next
            off_next += K * nch * BLK
            want_b = np.zeros((K, nch, 8, s, CW), np.int16)
            want_h = np.zeros((K, nch, 8, s, CW), np.int16)
            for r, hi in enumerate(rows):
                if (ho, hi) not in ext:
                    continue
                dlo, dhi, vb, vh = ext[(ho, hi)]
                for c in range(nch):
                    for p in range(s):
                        y = np.arange(CW)
                        d = s * (MW + TQ - 1 - 64 * c - y) + p
                        ok = (d >= dlo) & (d <= dhi)
                        want_b[:, c, r, p, y[ok]] = vb[d[ok] - dlo].T
                        want_h[:, c, r, p, y[ok]] = vh[d[ok] - dlo].T
            for t, (tab, want) in enumerate(((gtab, want_b), (gtab_h, want_h))):
                got = tab[off:off + K * nch * BLK].reshape(K, nch, 8, s, CW)
                assert np.array_equal(got, want), (z, ho, t)
    assert off_next == psi.c.ngtab


@pytest.mark.parametrize("case", [CASES[0], CASES[3], CASES[-1]], ids=lambda c: f"{c[0]}->{c[1]}")
def test_export_uniform_kpacked(lib, case):
    """The page's uniform K-packed form: counts and indices bit-exact against
    the oracle's union layout, values bit-exact against the built union
    values, zero padding, and nbr_pad < max_row rejected."""
    gi, go, kind, nrad, cut = case
    ref = oracle.build_psi(gi, go, kind, nrad, cut)
    psi = lib.Psi(gi, go, kind, nrad, cut)
    Ho, Kp = go[0], psi.c.K_pad
    counts = np.diff(ref.row_ptr)
    assert psi.c.max_row == counts.max()
    val = psi.tensor("val").cpu().numpy()
    for pad in (int(counts.max()), int(counts.max()) + 5):
        pidx = torch.full((Ho, pad, 2), -7, dtype=torch.int64, device="cuda")
        pval = torch.full((Ho, pad, Kp), float("nan"), dtype=torch.float32, device="cuda")
        pcnt = torch.full((Ho,), -7, dtype=torch.int64, device="cuda")
        lib.disco_psi_export_kpacked(psi.c, pidx, pval, pcnt, pad)
        torch.cuda.synchronize()
        pidx, pval, pcnt = pidx.cpu().numpy(), pval.cpu().numpy(), pcnt.cpu().numpy()
        assert np.array_equal(pcnt, counts)
        for ho in range(Ho):
            lo, hi_, n = ref.row_ptr[ho], ref.row_ptr[ho + 1], counts[ho]
            assert np.array_equal(pidx[ho, :n], ref.idx[lo:hi_])
            assert np.array_equal(pval[ho, :n], val[lo:hi_])
            assert not pidx[ho, n:].any() and not pval[ho, n:].any()
    with pytest.raises(lib.DiscoError) as e:
        lib.disco_psi_export_kpacked(psi.c, pidx_d := torch.zeros(1, dtype=torch.int64, device="cuda"),
                                     torch.zeros(1, device="cuda"), pidx_d, int(counts.max()) - 1)
    assert e.value.status == -1
