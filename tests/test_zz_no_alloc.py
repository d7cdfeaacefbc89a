"""The allocation-free input-gradient entry point.

disco_fused_conv_bwd_input_noalloc serves callers that cannot allocate device
memory themselves (a runtime whose allocator owns all device memory, or a hot
loop that must not risk cudaMalloc's implicit device synchronisation).  It
keeps dX in the library's fixed device scratch instead of a caller workspace.
This file is collected last on purpose: it checks, through the C ABI, that
the variant gives bit for bit the workspace entry point's result on two calls
in a row (the scratch keeps the previous call's contents; bf16 and fp16),
that the first call is within the suite's bar of the fp64 oracle, and that
oversized problems are rejected before any launch.  It needs nothing
from the other test files, so it also passes alone in a fresh process.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from tests._helpers import TOL, rel_err, to_np32

pytestmark = pytest.mark.gpu
BF = torch.bfloat16


@pytest.fixture(scope="module")
def lib():
    from sparse_spherical_convolution_gb300 import build
    build.build()
    import sparse_spherical_convolution_gb300 as d
    return d


CASES = [
    # (grid_in, grid_out, kind, nrad, cutoff, B, Cin, Cout, dtype)
    ((64, 128, 0), (64, 128, 0), 0, 5, 3 * math.pi / 64, 2, 32, 48, BF),     # CUDA-core dX GEMM
    ((128, 256, 0), (64, 128, 0), 1, 3, 3 * math.pi / 64, 1, 32, 64, BF),    # tensor-core dX GEMM + transpose
    ((128, 256, 0), (64, 128, 0), 1, 3, 3 * math.pi / 64, 1, 64, 64, torch.float16),  # fp16: Cin*K % 64 == 0
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: f"{c[0]}->{c[1]}-{str(c[8])[6:]}")
def test_noalloc_matches_workspace_entry_point_twice(lib, case):
    gi, go, kind, nrad, cut, B, Cin, Cout, dt = case
    psi = lib.Psi(gi, go, kind, nrad, cut)
    K = psi.c.K
    g = torch.Generator().manual_seed(21)
    W = (torch.randn((Cout, Cin, K), generator=g) / math.sqrt(Cin * K)).to(dt).cuda()
    ref = oracle.build_psi(gi, go, kind, nrad, cut)
    ws = torch.empty(lib.disco_fused_conv_bwd_input_workspace_bytes(psi.c, B, Cin, _CODE[dt]),
                     dtype=torch.uint8, device="cuda")
    for call in range(2):  # two calls in a row with different inputs
        dy = torch.randn((B, Cout, go[0], go[1]), generator=g).to(dt).cuda()
        want = torch.empty((B, Cin, gi[0], gi[1]), dtype=dt, device="cuda")
        got = torch.full((B, Cin, gi[0], gi[1]), float("nan"), dtype=dt, device="cuda")
        lib.disco_fused_conv_bwd_input(psi.c, dy, W, want, B, Cin, Cout, ws)
        lib.disco_fused_conv_bwd_input_noalloc(psi.c, dy, W, got, B, Cin, Cout)
        torch.cuda.synchronize()
        assert lib.disco_device_status() == 0
        # the same kernels on the same inputs: bit for bit the workspace result
        assert torch.equal(got, want), call
        if call == 0:  # and within the suite's bar of the fp64 oracle
            gxo, S = oracle.fused_bwd_input(ref, to_np32(dy), to_np32(W))
            assert rel_err(to_np32(got), gxo, S) <= TOL[dt]


_CODE = {BF: 1, torch.float16: 2}


def test_noalloc_rejects_problems_beyond_the_fixed_scratch(lib):
    gi, go = (361, 720, 1), (361, 720, 1)
    psi = lib.Psi(gi, go, 1, 3, 4 * math.pi / 360)
    B, Cin, Cout = 1, 64, 16   # dX = 64 * 9 * 361 * 720 * 2 bytes = 299 MB > 64 MiB
    assert lib.disco_fused_conv_bwd_input_workspace_bytes(psi.c, B, Cin) > lib.NOALLOC_SCRATCH_BYTES
    dy = torch.zeros((B, Cout, 361, 720), dtype=BF, device="cuda")
    W = torch.zeros((Cout, Cin, 9), dtype=BF, device="cuda")
    gx = torch.full((B, Cin, 361, 720), 7.0, dtype=BF, device="cuda")
    with pytest.raises(lib.DiscoError) as e:
        lib.disco_fused_conv_bwd_input_noalloc(psi.c, dy, W, gx, B, Cin, Cout)
    assert e.value.status == -7 and "scratch" in str(e.value)
    torch.cuda.synchronize()
    assert torch.all(gx == 7.0)  # nothing was launched
