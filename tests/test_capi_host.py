"""Host-side checks of the C ABI that need no GPU: the library builds, loads
and exports every symbol include/disco.h declares; host-only validation
returns the documented status without touching a device."""
import ctypes
import math
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from sparse_spherical_convolution_gb300 import build
    build.build()
    import sparse_spherical_convolution_gb300 as d
    return d


def _declared_functions():
    src = open(os.path.join(ROOT, "include", "disco.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(disco_[a-z0-9_]+)\s*\(", src)))


def test_exports_every_declared_symbol(lib):
    declared = _declared_functions()
    assert declared, "no declarations found"
    so = ctypes.CDLL(lib.library_path())
    for name in declared:
        assert hasattr(so, name), name
    assert set(declared) == set(lib.EXPORTED_SYMBOLS)


def test_bounds_checked_build_exports_the_same_symbols(lib):
    """The bounds-checked build (-DDISCO_DEBUG_BOUNDS) compiles from the same
    sources, exports the same symbols and says which build it is."""
    from sparse_spherical_convolution_gb300 import build
    path = build.build(debug_bounds=True)
    assert path == build.LIB_BOUNDS and path != build.LIB
    so = ctypes.CDLL(path)
    for name in _declared_functions():
        assert hasattr(so, name), name
    so.disco_build_flags.restype = ctypes.c_int32
    assert so.disco_build_flags() == lib.DISCO_BUILD_DEBUG_BOUNDS
    assert lib.disco_build_flags() == 0


def test_version_and_error_string(lib):
    assert lib.disco_version() >= 100
    assert isinstance(lib.disco_last_error(), str)


def test_workspace_bytes_host_validation(lib):
    b = lib.disco_basis(1, 3, 3 * math.pi / 64)
    n = lib.disco_psi_workspace_bytes((128, 256, 0), (64, 128, 0), b)
    assert n > 0 and n % 256 == 0
    with pytest.raises(lib.DiscoError) as e:
        lib.disco_psi_workspace_bytes((128, 250, 0), (64, 128, 0), b)   # W_in % W_out != 0
    assert e.value.status == -2
    with pytest.raises(lib.DiscoError) as e:
        lib.disco_psi_workspace_bytes((128, 256, 0), (64, 128, 0), lib.disco_basis(1, 6, 0.1))  # K = 18
    assert e.value.status == -2
    with pytest.raises(lib.DiscoError) as e:
        lib.disco_psi_workspace_bytes((128, 256, 0), (64, 128, 0), lib.disco_basis(0, 3, -1.0))
    assert e.value.status == -1
    with pytest.raises(lib.DiscoError) as e:
        lib.disco_psi_workspace_bytes((2, 8, 1), (2, 8, 1), lib.disco_basis(0, 3, 0.5))  # pole grid nlat < 3
    assert e.value.status == -1
    # Legendre-Gauss grids (poles = 2) are accepted, from 2 rows; other grid kinds are not
    assert lib.disco_psi_workspace_bytes((2, 8, 2), (2, 8, 2), lib.disco_basis(0, 3, 0.5)) > 0
    assert lib.disco_psi_workspace_bytes((721, 1440, 1), (360, 720, 2), b) > 0
    for bad in (3, -1):
        with pytest.raises(lib.DiscoError) as e:
            lib.disco_psi_workspace_bytes((16, 32, bad), (16, 32, 0), b)
        assert e.value.status == -1


def test_hot_calls_reject_unbuilt_psi_before_any_launch(lib):
    empty = lib.disco_psi()
    so = lib.load_library()
    assert so.disco_fwd(ctypes.byref(empty), None, None, 1, 1, 1, None) == -1
    assert "psi" in lib.disco_last_error()
    assert so.disco_bwd(None, None, None, 1, 1, 1, None) == -1
    assert so.disco_fused_conv(ctypes.byref(empty), None, None, None, 1, 16, 16, 1, None, 0, None) == -1
    assert so.disco_fused_conv_bwd_input(ctypes.byref(empty), None, None, None, 1, 16, 16, 1,
                                         None, 0, None) == -1


def test_binding_rejects_host_tensors_before_the_library(lib):
    """The binding checks device, dtype and size in Python first: a CPU tensor
    never reaches a kernel (this runs without a GPU)."""
    import torch
    psi = lib.disco_psi()
    psi.grid_in = lib.disco_grid(8, 16, 0)
    psi.grid_out = lib.disco_grid(8, 16, 0)
    psi.K = 3
    x = torch.zeros((1, 2, 8, 16), dtype=torch.float32)
    X = torch.zeros((1, 2, 3, 8, 16), dtype=torch.float32)
    with pytest.raises(lib.DiscoError) as e:
        lib.disco_fwd(psi, x, X, 1, 2)
    assert e.value.status == -1 and "CUDA device" in str(e.value)
    with pytest.raises(lib.DiscoError) as e:
        lib.disco_fwd_host(psi, x, X[:, :1], 1, 2, None)
    assert e.value.status == -1 and "elements" in str(e.value)
