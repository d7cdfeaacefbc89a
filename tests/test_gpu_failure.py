"""Failure detection without a GPU fault: a bounded mbarrier wait that
nothing completes runs out, sets its status bit, and the context stays
usable (the next contraction runs and is correct)."""
import math

import numpy as np
import pytest
import torch

import oracle
from tests._helpers import TOL, rel_err, to_np32

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    from sparse_spherical_convolution_gb300 import build
    build.build()
    import sparse_spherical_convolution_gb300 as d
    d.disco_device_status(clear=True)
    return d


def test_timed_out_wait_reaches_status_and_context_survives(lib):
    assert lib.disco_device_status(clear=True) == 0
    lib.disco_check_wait_timeout(1 << 12)
    assert lib.disco_device_status(clear=False) == 16
    assert lib.disco_device_status(clear=True) == 16  # read again, then cleared
    assert lib.disco_device_status() == 0
    # the context still works: a tensor-core contraction right after
    gi = go = (64, 128, 0)
    ref = oracle.build_psi(gi, go, 0, 5, 3 * math.pi / 64)
    psi = lib.Psi(gi, go, 0, 5, 3 * math.pi / 64)
    g = torch.Generator().manual_seed(41)
    x = torch.randn((1, 16, 64, 128), generator=g).to(torch.bfloat16)
    X = torch.empty((1, 16, ref.K, 64, 128), dtype=torch.bfloat16, device="cuda")
    lib.disco_fwd(psi.c, x.cuda(), X, 1, 16)
    torch.cuda.synchronize()
    assert lib.disco_device_status() == 0
    Xo, S = oracle.fwd(ref, to_np32(x))
    assert rel_err(to_np32(X), Xo, S) <= TOL[torch.bfloat16]


def test_wait_check_rejects_bad_limits(lib):
    for bad in (0, (1 << 24) + 1):
        with pytest.raises(lib.DiscoError) as e:
            lib.disco_check_wait_timeout(bad)
        assert e.value.status == -1


def _foreign_tag_case(lib, fwd: bool):
    """The scheduler word of the next persistent launch holds another
    launch's tag with its counter part-way (as every earlier launch leaves
    it): the launch takes the word over and computes every tile."""
    gi = go = (64, 128, 0)
    ref = oracle.build_psi(gi, go, 0, 5, 3 * math.pi / 64)
    psi = lib.Psi(gi, go, 0, 5, 3 * math.pi / 64)
    g = torch.Generator().manual_seed(43)
    B, C = 1, 130
    x = torch.randn((B, C, 64, 128), generator=g).to(torch.bfloat16).cuda()
    G = torch.randn((B, C, ref.K, 64, 128), generator=g).to(torch.bfloat16).cuda()
    inp, shape = (x, (B, C, ref.K, 64, 128)) if fwd else (G, (B, C, 64, 128))
    call = lib.disco_fwd if fwd else lib.disco_bwd
    assert lib.disco_device_status(clear=True) == 0
    out = torch.full(shape, 3.0, dtype=torch.bfloat16, device="cuda")
    lib.disco_check_sched_takeover()   # also walks the protocol on a private word
    call(psi.c, inp, out, B, C)
    assert lib.disco_device_status() == 0
    if fwd:
        want, S = oracle.fwd(ref, to_np32(x))
    else:
        want, S = oracle.bwd(ref, to_np32(G))
    assert rel_err(to_np32(out), want, S) <= TOL[torch.bfloat16]
    out2 = torch.full(shape, 3.0, dtype=torch.bfloat16, device="cuda")
    call(psi.c, inp, out2, B, C)   # the launch after it draws from its own word as usual
    assert lib.disco_device_status() == 0
    assert torch.equal(out, out2)


def test_foreign_scheduler_tag_is_taken_over_forward(lib):
    _foreign_tag_case(lib, True)


def test_foreign_scheduler_tag_is_taken_over_transpose(lib):
    _foreign_tag_case(lib, False)


def test_scheduler_words_reused_across_many_launches(lib):
    """Many more persistent launches than the scheduler tables have words
    (1024 per kernel family; launch ids are shared by the families, so
    alternating forward and transpose launches each reuse every other word),
    on two streams at once: words are taken over again and again while
    launches on the other stream draw from theirs.  Every result must equal
    the one computed alone, bit for bit, with a clean status word."""
    gi = go = (64, 128, 0)
    psi = lib.Psi(gi, go, 0, 5, 3 * math.pi / 64)
    B, C, K = 1, 130, psi.c.K
    g = torch.Generator(device="cuda").manual_seed(17)
    x = torch.randn((B, C, 64, 128), generator=g, device="cuda").to(torch.bfloat16)
    G = torch.randn((B, C, K, 64, 128), generator=g, device="cuda").to(torch.bfloat16)
    X0 = torch.empty((B, C, K, 64, 128), dtype=torch.bfloat16, device="cuda")
    gx0 = torch.empty_like(x)
    lib.disco_fwd(psi.c, x, X0, B, C)
    lib.disco_bwd(psi.c, G, gx0, B, C)
    torch.cuda.synchronize()
    assert lib.disco_device_status(clear=True) == 0
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    Xs = [torch.empty_like(X0) for _ in range(2)]
    gxs = [torch.empty_like(gx0) for _ in range(2)]
    for i in range(1100):  # 2200 persistent launches, alternating streams
        st = s1 if i % 2 == 0 else s2
        lib.disco_fwd(psi.c, x, Xs[i % 2], B, C, stream=st)
        lib.disco_bwd(psi.c, G, gxs[i % 2], B, C, stream=st)
    torch.cuda.synchronize()
    assert lib.disco_device_status(clear=True) == 0
    for X, gx in zip(Xs, gxs):
        assert torch.equal(X, X0) and torch.equal(gx, gx0)
