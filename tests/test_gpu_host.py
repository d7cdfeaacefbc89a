"""Host-buffer entry points (disco_fwd_host / disco_bwd_host): the same
results as the device entry points bit for bit, on ragged block counts,
pinned and pageable memory, fp32 / bf16 / fp16, two calls in flight on two
streams, and the workspace rule."""
import math

import pytest
import torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    from sparse_spherical_convolution_gb300 import build
    build.build()
    import sparse_spherical_convolution_gb300 as d
    d.disco_device_status(clear=True)
    return d


# (grid_in, grid_out, kind, nrad, cutoff, B, C, dtype)
CASES = [
    ((64, 128, 0), (64, 128, 0), 0, 5, 3 * math.pi / 64, 2, 70, torch.bfloat16),     # 140 planes: 2 blocks, ragged
    ((128, 256, 0), (64, 128, 0), 1, 3, 3 * math.pi / 64, 3, 100, torch.float16),    # 300 planes: 3 blocks
    ((16, 32, 0), (16, 32, 0), 0, 3, 2 * math.pi / 16, 1, 2, torch.float32),         # one small block
    ((361, 720, 1), (361, 720, 1), 1, 3, 4 * math.pi / 360, 2, 128, torch.bfloat16), # the 361x720 workload
]


def _device_ref(lib, psi, x, G, B, C):
    X = torch.empty(G.shape, dtype=x.dtype, device="cuda")
    gx = torch.empty(x.shape, dtype=x.dtype, device="cuda")
    lib.disco_fwd(psi.c, x.cuda(), X, B, C)
    lib.disco_bwd(psi.c, G.cuda(), gx, B, C)
    torch.cuda.synchronize()
    return X.cpu(), gx.cpu()


@pytest.mark.parametrize("pinned", [True, False])
@pytest.mark.parametrize("case", CASES, ids=lambda c: f"{c[0]}->{c[1]}-B{c[5]}C{c[6]}-{str(c[7])[6:]}")
def test_host_entry_points_match_device(lib, case, pinned):
    gi, go, kind, nrad, cut, B, C, dt = case
    psi = lib.Psi(gi, go, kind, nrad, cut)
    K = psi.c.K
    g = torch.Generator().manual_seed(51)
    x = torch.randn((B, C, gi[0], gi[1]), generator=g).to(dt)
    G = torch.randn((B, C, K, go[0], go[1]), generator=g).to(dt)
    Xd, gxd = _device_ref(lib, psi, x, G, B, C)
    if pinned:
        x, G = x.pin_memory(), G.pin_memory()
    Xh = torch.full(G.shape, float("nan"), dtype=dt, pin_memory=pinned)
    gxh = torch.full(x.shape, float("nan"), dtype=dt, pin_memory=pinned)
    code = {torch.float32: lib.DISCO_F32, torch.bfloat16: lib.DISCO_BF16, torch.float16: lib.DISCO_F16}[dt]
    wf = torch.empty(lib.disco_host_workspace_bytes(psi.c, B, C, True, code), dtype=torch.uint8, device="cuda")
    wb = torch.empty(lib.disco_host_workspace_bytes(psi.c, B, C, False, code), dtype=torch.uint8, device="cuda")
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    lib.disco_fwd_host(psi.c, x, Xh, B, C, wf, s1)   # both calls in flight at once
    lib.disco_bwd_host(psi.c, G, gxh, B, C, wb, s2)
    s1.synchronize()
    s2.synchronize()
    assert lib.disco_device_status() == 0
    assert torch.equal(Xh, Xd) and torch.equal(gxh, gxd)


def test_host_workspace_rule(lib):
    psi = lib.Psi((64, 128, 0), (64, 128, 0), 0, 5, 3 * math.pi / 64)
    x = torch.zeros((1, 4, 64, 128), dtype=torch.bfloat16)
    X = torch.zeros((1, 4, psi.c.K, 64, 128), dtype=torch.bfloat16)
    need = lib.disco_host_workspace_bytes(psi.c, 1, 4, True, lib.DISCO_BF16)
    assert need > 0
    small = torch.empty(need - 256, dtype=torch.uint8, device="cuda")
    with pytest.raises(lib.DiscoError) as e:
        lib.disco_fwd_host(psi.c, x, X, 1, 4, small)
    assert e.value.status == -7


def test_binding_rejects_wrong_device_dtype_and_size(lib):
    """The binding refuses host tensors, mixed dtypes and wrong element counts
    before calling the library; the C ABI itself refuses host pointers."""
    import ctypes
    psi = lib.Psi((64, 128, 0), (64, 128, 0), 0, 5, 3 * math.pi / 64)
    K = psi.c.K
    x = torch.zeros((1, 4, 64, 128), dtype=torch.bfloat16, device="cuda")
    X = torch.full((1, 4, K, 64, 128), 5.0, dtype=torch.bfloat16, device="cuda")
    for bad_x, bad_X in [(x.cpu(), X), (x, X.float()), (x, X[:, :3]), (x[:, :3], X)]:
        with pytest.raises(lib.DiscoError) as e:
            lib.disco_fwd(psi.c, bad_x.contiguous(), bad_X.contiguous(), 1, 4)
        assert e.value.status == -1
    W = torch.zeros((8, 4, K), dtype=torch.float16, device="cuda")
    y = torch.zeros((1, 8, 64, 128), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(lib.DiscoError):
        lib.disco_fused_conv(psi.c, x, W, y, 1, 4, 8)      # W of another dtype
    # through the C ABI: a host buffer as X is refused on the host
    so = lib.load_library()
    host = (ctypes.c_uint16 * X.numel())()
    st = so.disco_fwd(ctypes.byref(psi.c), ctypes.c_void_p(x.data_ptr()), ctypes.cast(host, ctypes.c_void_p),
                      1, 4, lib.DISCO_BF16, None)
    assert st == -1 and "device memory" in lib.disco_last_error()
    torch.cuda.synchronize()
    assert torch.all(X == 5.0)
