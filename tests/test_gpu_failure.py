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
