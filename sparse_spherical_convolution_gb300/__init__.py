"""GB300 (sm_103a) DISCO convolution on the sphere: Python binding of the C ABI.

The binding only marshals arguments: every step runs in the CUDA library
``_build/libdisco_gb300_<arch>.so`` (built by ``build.py``).  If the library
is missing, importing the functions raises; there is no fallback.

The functions carry the names of the C ABI (``include/disco.h``) and take
torch tensors for device memory; torch's current CUDA stream is used unless a
stream is given.
"""
from __future__ import annotations

import ctypes
import os

from . import build as _build_mod

__all__ = [
    "DiscoError", "disco_grid", "disco_basis", "disco_run", "disco_psi", "Psi",
    "disco_version", "disco_build_flags", "DISCO_BUILD_DEBUG_BOUNDS", "DISCO_ERR_DEVICE_BOUNDS",
    "disco_last_error", "disco_psi_workspace_bytes", "disco_psi_plan",
    "disco_build_psi_kpacked", "disco_psi_export_kpacked", "disco_check_wait_timeout", "disco_fwd", "disco_bwd",
    "disco_host_workspace_bytes", "disco_fwd_host", "disco_bwd_host",
    "disco_fused_conv_workspace_bytes",
    "disco_fused_conv", "disco_fused_conv_bwd_input_workspace_bytes", "disco_fused_conv_bwd_input",
    "disco_fused_conv_bwd_input_noalloc", "disco_fused_conv_bwd_weight_workspace_bytes",
    "disco_fused_conv_bwd_weight", "disco_device_status", "disco_check_sched_takeover", "library_path",
    "load_library", "EXPORTED_SYMBOLS", "NOALLOC_SCRATCH_BYTES",
]

NOALLOC_SCRATCH_BYTES = 64 << 20

DISCO_F32, DISCO_BF16, DISCO_F16 = 0, 1, 2

EXPORTED_SYMBOLS = [
    "disco_version", "disco_last_error", "disco_psi_workspace_bytes", "disco_psi_plan",
    "disco_build_psi_kpacked", "disco_fwd", "disco_bwd", "disco_fused_conv_workspace_bytes",
    "disco_fused_conv", "disco_fused_conv_bwd_input_workspace_bytes", "disco_fused_conv_bwd_input",
    "disco_fused_conv_bwd_input_noalloc", "disco_fused_conv_bwd_weight_workspace_bytes",
    "disco_fused_conv_bwd_weight", "disco_device_status", "disco_psi_export_kpacked",
    "disco_check_wait_timeout", "disco_host_workspace_bytes", "disco_fwd_host", "disco_bwd_host",
    "disco_check_sched_takeover", "disco_build_flags",
]


class DiscoError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"disco status {status}: {message}")
        self.status = status


class disco_grid(ctypes.Structure):
    _fields_ = [("nlat", ctypes.c_int32), ("nlon", ctypes.c_int32), ("poles", ctypes.c_int32)]


class disco_basis(ctypes.Structure):
    _fields_ = [("kind", ctypes.c_int32), ("n_radial", ctypes.c_int32), ("cutoff", ctypes.c_double)]


class disco_run(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in ("ho", "hi", "D", "hoff", "e0", "len", "npair", "anti")]


_PSI_ARRAYS = ["row_ptr", "idx", "val", "csr_row_ptr", "csr_col", "csr_val", "run_ptr", "runs",
               "trun_ptr", "truns", "hval", "row_order", "ftab_off", "ftab", "grp_ptr", "grp", "gtab",
               "ftab_h", "gtab_h"]


class disco_psi(ctypes.Structure):
    _fields_ = [("grid_in", disco_grid), ("grid_out", disco_grid), ("basis", disco_basis),
                ("K", ctypes.c_int32), ("K_pad", ctypes.c_int32), ("s", ctypes.c_int32),
                ("max_row", ctypes.c_int32), ("nnz", ctypes.c_int64), ("nnz_csr", ctypes.c_int64),
                ("nruns", ctypes.c_int64), ("nhval", ctypes.c_int64), ("nftab", ctypes.c_int64),
                ("ngrp", ctypes.c_int32), ("grp_max", ctypes.c_int32), ("ngrp_ent", ctypes.c_int64),
                ("ngtab", ctypes.c_int64), ("bytes", ctypes.c_size_t)] + \
               [(n, ctypes.c_void_p) for n in _PSI_ARRAYS]


_lib = None


def library_path() -> str:
    """The product library, or its bounds-checked build when the environment
    sets DISCO_GB300_BOUNDS_CHECKED=1 (a diagnostic build, see build.py)."""
    if os.environ.get("DISCO_GB300_BOUNDS_CHECKED") == "1":
        return _build_mod.LIB_BOUNDS
    return _build_mod.LIB


def load_library():
    """Loads the built library; raises if it is missing (no fallback path)."""
    global _lib
    if _lib is not None:
        return _lib
    path = library_path()
    if not os.path.exists(path):
        raise RuntimeError(f"DISCO CUDA library not built: {path} is missing "
                           "(run `python -m sparse_spherical_convolution_gb300.build`)")
    lib = ctypes.CDLL(path)
    P, I32, SZ = ctypes.c_void_p, ctypes.c_int32, ctypes.c_size_t
    PG, PB, PP = ctypes.POINTER(disco_grid), ctypes.POINTER(disco_basis), ctypes.POINTER(disco_psi)
    lib.disco_version.restype = I32
    lib.disco_version.argtypes = []
    lib.disco_build_flags.restype = I32
    lib.disco_build_flags.argtypes = []
    lib.disco_last_error.restype = ctypes.c_char_p
    lib.disco_last_error.argtypes = []
    lib.disco_psi_workspace_bytes.restype = ctypes.c_int
    lib.disco_psi_workspace_bytes.argtypes = [PG, PG, PB, ctypes.POINTER(SZ)]
    lib.disco_psi_plan.restype = ctypes.c_int
    lib.disco_psi_plan.argtypes = [PG, PG, PB, P, SZ, P, PP]
    lib.disco_build_psi_kpacked.restype = ctypes.c_int
    lib.disco_build_psi_kpacked.argtypes = [PP, P, SZ, P, SZ, P]
    lib.disco_host_workspace_bytes.restype = SZ
    lib.disco_host_workspace_bytes.argtypes = [PP, I32, I32, I32, ctypes.c_int]
    for nm in ("disco_fwd_host", "disco_bwd_host"):
        getattr(lib, nm).restype = ctypes.c_int
        getattr(lib, nm).argtypes = [PP, P, P, I32, I32, ctypes.c_int, P, SZ, P]
    lib.disco_check_wait_timeout.restype = ctypes.c_int
    lib.disco_check_wait_timeout.argtypes = [ctypes.c_uint32, P]
    lib.disco_check_sched_takeover.restype = ctypes.c_int
    lib.disco_check_sched_takeover.argtypes = []
    lib.disco_psi_export_kpacked.restype = ctypes.c_int
    lib.disco_psi_export_kpacked.argtypes = [PP, P, P, P, I32, P]
    lib.disco_fwd.restype = ctypes.c_int
    lib.disco_fwd.argtypes = [PP, P, P, I32, I32, ctypes.c_int, P]
    lib.disco_bwd.restype = ctypes.c_int
    lib.disco_bwd.argtypes = [PP, P, P, I32, I32, ctypes.c_int, P]
    lib.disco_fused_conv_workspace_bytes.restype = SZ
    lib.disco_fused_conv_workspace_bytes.argtypes = [PP, I32, I32, I32, ctypes.c_int]
    lib.disco_fused_conv.restype = ctypes.c_int
    lib.disco_fused_conv.argtypes = [PP, P, P, P, I32, I32, I32, ctypes.c_int, P, SZ, P]
    lib.disco_fused_conv_bwd_input_workspace_bytes.restype = SZ
    lib.disco_fused_conv_bwd_input_workspace_bytes.argtypes = [PP, I32, I32, ctypes.c_int]
    lib.disco_fused_conv_bwd_input.restype = ctypes.c_int
    lib.disco_fused_conv_bwd_input.argtypes = [PP, P, P, P, I32, I32, I32, ctypes.c_int, P, SZ, P]
    lib.disco_fused_conv_bwd_input_noalloc.restype = ctypes.c_int
    lib.disco_fused_conv_bwd_input_noalloc.argtypes = [PP, P, P, P, I32, I32, I32, ctypes.c_int, P]
    lib.disco_fused_conv_bwd_weight_workspace_bytes.restype = SZ
    lib.disco_fused_conv_bwd_weight_workspace_bytes.argtypes = [PP, I32, I32, I32, ctypes.c_int]
    lib.disco_fused_conv_bwd_weight.restype = ctypes.c_int
    lib.disco_fused_conv_bwd_weight.argtypes = [PP, P, P, P, I32, I32, I32, ctypes.c_int, P, SZ, P]
    lib.disco_device_status.restype = ctypes.c_int
    lib.disco_device_status.argtypes = [ctypes.POINTER(I32), I32]
    _lib = lib
    return lib


def _check(status: int):
    if status != 0:
        raise DiscoError(status, load_library().disco_last_error().decode())


def _stream(stream):
    import torch
    if stream is None:
        return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, int):
        return ctypes.c_void_p(stream)
    return ctypes.c_void_p(stream.cuda_stream)


def _dtype(t) -> int:
    import torch
    if t.dtype == torch.float32:
        return DISCO_F32
    if t.dtype == torch.bfloat16:
        return DISCO_BF16
    if t.dtype == torch.float16:
        return DISCO_F16
    raise DiscoError(-2, f"unsupported dtype {t.dtype}")


def _ptr(t):
    if t is None:
        return None
    if not t.is_contiguous():
        raise DiscoError(-1, "tensors must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


def _dev(t, name: str, numel: int, dtype=None):
    """Pointer of a device tensor after checking it: on the current CUDA
    device, contiguous, `numel` elements, and of `dtype` when given.  A
    mismatch raises DiscoError(-1) before any call into the library."""
    import torch
    if t is None:
        raise DiscoError(-1, f"{name} is None")
    if not t.is_cuda or t.device.index != torch.cuda.current_device():
        raise DiscoError(-1, f"{name} must be a tensor on the current CUDA device, got {t.device}")
    if dtype is not None and t.dtype != dtype:
        raise DiscoError(-1, f"{name} has dtype {t.dtype}, the call's dtype is {dtype}")
    if t.numel() != int(numel):
        raise DiscoError(-1, f"{name} has {t.numel()} elements, the call needs {int(numel)}")
    return _ptr(t)


def _host(t, name: str, numel: int, dtype=None):
    """Pointer of a host (CPU) tensor after the same checks as _dev."""
    if t is None or t.is_cuda:
        raise DiscoError(-1, f"{name} must be a CPU tensor")
    if dtype is not None and t.dtype != dtype:
        raise DiscoError(-1, f"{name} has dtype {t.dtype}, the call's dtype is {dtype}")
    if t.numel() != int(numel):
        raise DiscoError(-1, f"{name} has {t.numel()} elements, the call needs {int(numel)}")
    return _ptr(t)


def _ws(t, name: str = "workspace"):
    """(pointer, bytes) of an optional device workspace."""
    import torch
    if t is None:
        return None, 0
    if not t.is_cuda or t.device.index != torch.cuda.current_device():
        raise DiscoError(-1, f"{name} must be a tensor on the current CUDA device")
    return _ptr(t), t.numel() * t.element_size()


def _sizes(psi):
    """(H_in*W_in, K*H_out*W_out, H_out*W_out, K) of a built psi."""
    pin = psi.grid_in.nlat * psi.grid_in.nlon
    pout = psi.grid_out.nlat * psi.grid_out.nlon
    return pin, psi.K * pout, pout, psi.K


# ------------------------------------------------------------------ ABI calls

def disco_version() -> int:
    return load_library().disco_version()


DISCO_BUILD_DEBUG_BOUNDS = 1
DISCO_ERR_DEVICE_BOUNDS = -8


def disco_build_flags() -> int:
    """DISCO_BUILD_DEBUG_BOUNDS when the loaded library is the bounds-checked build."""
    return load_library().disco_build_flags()


def disco_last_error() -> str:
    return load_library().disco_last_error().decode()


def _grid(g) -> disco_grid:
    return g if isinstance(g, disco_grid) else disco_grid(*[int(v) for v in g])


def _basis(kind, n_radial=None, cutoff=None) -> disco_basis:
    if isinstance(kind, disco_basis):
        return kind
    return disco_basis(int(kind), int(n_radial), float(cutoff))


def disco_psi_workspace_bytes(grid_in, grid_out, basis) -> int:
    n = ctypes.c_size_t()
    _check(load_library().disco_psi_workspace_bytes(
        ctypes.byref(_grid(grid_in)), ctypes.byref(_grid(grid_out)), ctypes.byref(basis),
        ctypes.byref(n)))
    return n.value


def disco_psi_plan(grid_in, grid_out, basis, workspace, stream=None) -> disco_psi:
    psi = disco_psi()
    _check(load_library().disco_psi_plan(
        ctypes.byref(_grid(grid_in)), ctypes.byref(_grid(grid_out)), ctypes.byref(basis),
        *_ws(workspace), _stream(stream), ctypes.byref(psi)))
    return psi


def disco_build_psi_kpacked(psi: disco_psi, buffer, workspace, stream=None) -> None:
    _check(load_library().disco_build_psi_kpacked(
        ctypes.byref(psi), *_ws(buffer, "buffer"), *_ws(workspace), _stream(stream)))


def disco_host_workspace_bytes(psi: disco_psi, B: int, C: int, forward: bool, dtype=DISCO_BF16) -> int:
    return load_library().disco_host_workspace_bytes(ctypes.byref(psi), B, C, 1 if forward else 0, dtype)


def disco_fwd_host(psi: disco_psi, x_host, X_host, B: int, C: int, workspace, stream=None) -> None:
    """x_host, X_host: CPU tensors (pinned for overlap); workspace: device."""
    pin, pX, _, _ = _sizes(psi)
    dt = x_host.dtype
    xp = _host(x_host, "x_host", B * C * pin, dt)
    Xp = _host(X_host, "X_host", B * C * pX, dt)
    wp, wn = _ws(workspace)
    _check(load_library().disco_fwd_host(ctypes.byref(psi), xp, Xp, B, C, _dtype(x_host), wp, wn,
                                         _stream(stream)))


def disco_bwd_host(psi: disco_psi, G_host, gx_host, B: int, C: int, workspace, stream=None) -> None:
    """G_host, gx_host: CPU tensors (pinned for overlap); workspace: device."""
    pin, pX, _, _ = _sizes(psi)
    dt = G_host.dtype
    Gp = _host(G_host, "G_host", B * C * pX, dt)
    gp = _host(gx_host, "gx_host", B * C * pin, dt)
    wp, wn = _ws(workspace)
    _check(load_library().disco_bwd_host(ctypes.byref(psi), Gp, gp, B, C, _dtype(G_host), wp, wn,
                                         _stream(stream)))


def disco_check_wait_timeout(limit: int, stream=None) -> None:
    _check(load_library().disco_check_wait_timeout(limit, _stream(stream)))


def disco_check_sched_takeover() -> None:
    """Walks the scheduler protocol, then leaves a foreign tag in the next launch's words (diagnostic)."""
    _check(load_library().disco_check_sched_takeover())


def disco_psi_export_kpacked(psi: disco_psi, pack_idx, pack_val, pack_count, nbr_pad: int,
                             stream=None) -> None:
    import torch
    H = psi.grid_out.nlat
    ip = _dev(pack_idx, "pack_idx", H * nbr_pad * 2, torch.int64)
    vp = _dev(pack_val, "pack_val", H * nbr_pad * psi.K_pad, torch.float32)
    cp = _dev(pack_count, "pack_count", H, torch.int64)
    _check(load_library().disco_psi_export_kpacked(ctypes.byref(psi), ip, vp, cp, nbr_pad, _stream(stream)))


def disco_fwd(psi: disco_psi, x, X, B: int, C: int, stream=None) -> None:
    pin, pX, _, _ = _sizes(psi)
    xp = _dev(x, "x", B * C * pin)
    Xp = _dev(X, "X", B * C * pX, x.dtype)
    _check(load_library().disco_fwd(ctypes.byref(psi), xp, Xp, B, C, _dtype(x), _stream(stream)))


def disco_bwd(psi: disco_psi, G, gx, B: int, C: int, stream=None) -> None:
    pin, pX, _, _ = _sizes(psi)
    Gp = _dev(G, "G", B * C * pX)
    gp = _dev(gx, "gx", B * C * pin, G.dtype)
    _check(load_library().disco_bwd(ctypes.byref(psi), Gp, gp, B, C, _dtype(G), _stream(stream)))


def disco_fused_conv_workspace_bytes(psi: disco_psi, B: int, Cin: int, Cout: int, dtype=DISCO_BF16) -> int:
    return load_library().disco_fused_conv_workspace_bytes(ctypes.byref(psi), B, Cin, Cout, dtype)


def disco_fused_conv(psi: disco_psi, x, W, y, B: int, Cin: int, Cout: int, workspace=None,
                     stream=None) -> None:
    pin, _, pout, K = _sizes(psi)
    xp = _dev(x, "x", B * Cin * pin)
    Wp = _dev(W, "W", Cout * Cin * K, x.dtype)
    yp = _dev(y, "y", B * Cout * pout, x.dtype)
    wp, wn = _ws(workspace)
    _check(load_library().disco_fused_conv(ctypes.byref(psi), xp, Wp, yp, B, Cin, Cout, _dtype(x), wp, wn,
                                           _stream(stream)))


def disco_fused_conv_bwd_input_workspace_bytes(psi: disco_psi, B: int, Cin: int, dtype=DISCO_BF16) -> int:
    return load_library().disco_fused_conv_bwd_input_workspace_bytes(ctypes.byref(psi), B, Cin, dtype)


def disco_fused_conv_bwd_input(psi: disco_psi, dy, W, gx, B: int, Cin: int, Cout: int,
                               workspace, stream=None) -> None:
    pin, _, pout, K = _sizes(psi)
    dp = _dev(dy, "dy", B * Cout * pout)
    Wp = _dev(W, "W", Cout * Cin * K, dy.dtype)
    gp = _dev(gx, "gx", B * Cin * pin, dy.dtype)
    wp, wn = _ws(workspace)
    _check(load_library().disco_fused_conv_bwd_input(ctypes.byref(psi), dp, Wp, gp, B, Cin, Cout, _dtype(dy),
                                                     wp, wn, _stream(stream)))


def disco_fused_conv_bwd_weight_workspace_bytes(psi: disco_psi, B: int, Cin: int, Cout: int,
                                                 dtype=DISCO_BF16) -> int:
    return load_library().disco_fused_conv_bwd_weight_workspace_bytes(ctypes.byref(psi), B, Cin, Cout, dtype)


def disco_fused_conv_bwd_weight(psi: disco_psi, x, dy, dW, B: int, Cin: int, Cout: int,
                                workspace, stream=None) -> None:
    pin, _, pout, K = _sizes(psi)
    xp = _dev(x, "x", B * Cin * pin)
    dp = _dev(dy, "dy", B * Cout * pout, x.dtype)
    Wp = _dev(dW, "dW", Cout * Cin * K, x.dtype)
    wp, wn = _ws(workspace)
    _check(load_library().disco_fused_conv_bwd_weight(ctypes.byref(psi), xp, dp, Wp, B, Cin, Cout, _dtype(x),
                                                      wp, wn, _stream(stream)))


def disco_fused_conv_bwd_input_noalloc(psi: disco_psi, dy, W, gx, B: int, Cin: int, Cout: int,
                                       stream=None) -> None:
    """disco_fused_conv_bwd_input without a workspace argument: the library's
    fixed device scratch holds dX (see include/disco.h for limits and rules)."""
    pin, _, pout, K = _sizes(psi)
    dp = _dev(dy, "dy", B * Cout * pout)
    Wp = _dev(W, "W", Cout * Cin * K, dy.dtype)
    gp = _dev(gx, "gx", B * Cin * pin, dy.dtype)
    _check(load_library().disco_fused_conv_bwd_input_noalloc(
        ctypes.byref(psi), dp, Wp, gp, B, Cin, Cout, _dtype(dy), _stream(stream)))


def disco_device_status(clear: bool = True) -> int:
    """Device status word (0 = no bounded wait timed out); synchronises the device.
    Raises DiscoError with status DISCO_ERR_DEVICE_BOUNDS when a range check
    of the bounds-checked build failed."""
    v = ctypes.c_int32()
    _check(load_library().disco_device_status(ctypes.byref(v), 1 if clear else 0))
    return v.value


# ------------------------------------------------------------ convenience

class Psi:
    """psi built on the device, with the torch buffers that own its memory.

    ``Psi(grid_in, grid_out, kind, n_radial, cutoff)`` runs disco_psi_plan and
    disco_build_psi_kpacked on the current CUDA device and stream."""

    _DT = {"row_ptr": "int32", "idx": "int32", "val": "float32", "csr_row_ptr": "int32",
           "csr_col": "int32", "csr_val": "float32", "run_ptr": "int32", "runs": "int32",
           "trun_ptr": "int32", "truns": "int32", "hval": "float32", "row_order": "int32",
           "ftab_off": "int32", "ftab": "int16", "grp_ptr": "int32", "grp": "int32", "gtab": "int16",
           "ftab_h": "int16", "gtab_h": "int16"}

    def __init__(self, grid_in, grid_out, kind: int, n_radial: int, cutoff: float, stream=None):
        import torch
        self.basis = _basis(kind, n_radial, cutoff)
        gi, go = _grid(grid_in), _grid(grid_out)
        wsb = disco_psi_workspace_bytes(gi, go, self.basis)
        self.workspace = torch.empty(max(wsb, 256), dtype=torch.uint8, device="cuda")
        self.c = disco_psi_plan(gi, go, self.basis, self.workspace, stream)
        self.buffer = torch.empty(max(self.c.bytes, 256), dtype=torch.uint8, device="cuda")
        disco_build_psi_kpacked(self.c, self.buffer, self.workspace, stream)

    def _sizes(self):
        c = self.c
        Hin, Hout = c.grid_in.nlat, c.grid_out.nlat
        return {"row_ptr": (Hout + 1,), "idx": (c.nnz, 2), "val": (c.nnz, c.K_pad),
                "csr_row_ptr": (c.K * Hout + 1,), "csr_col": (c.nnz_csr,),
                "csr_val": (c.nnz_csr,), "run_ptr": (Hout + 1,), "runs": (c.nruns, 8),
                "trun_ptr": (Hin + 1,), "truns": (c.nruns,), "hval": (c.nhval, c.K_pad),
                "row_order": (Hout,), "ftab_off": (c.nruns + 1,), "ftab": (c.nftab,),
                "grp_ptr": (c.ngrp + 1,), "grp": (c.ngrp_ent, 4), "gtab": (c.ngtab,),
                "ftab_h": (c.nftab,), "gtab_h": (c.ngtab,)}

    def tensor(self, name: str):
        """Device view of one psi array (for inspection and tests)."""
        import torch
        ptr = getattr(self.c, name)
        off = ptr - self.buffer.data_ptr()
        shape = self._sizes()[name]
        n = 1
        for v in shape:
            n *= int(v)
        dt = getattr(torch, self._DT[name])
        esz = torch.tensor([], dtype=dt).element_size()
        return self.buffer[off:off + n * esz].view(dt).view(*[int(v) for v in shape])
