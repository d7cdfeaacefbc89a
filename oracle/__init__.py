"""Plain fp64 CPU oracle for the DISCO convolution on the sphere.

TEST INFRASTRUCTURE ONLY: the tests, the smoke check and the CPU-baseline leg
of the benchmark may import this package; the product library never does.  It
shares no code with the CUDA path.  The arithmetic lives in ``disco_oracle.c``
(plain loops, fp64); this module only compiles it and marshals numpy arrays.

Pinned by the ``not gpu`` tests (dense brute force with independent vector
geometry, adjoint identity, longitude equivariance, the indicator-basis
neighbourhood sum, normalisation and symmetry invariants, hand-derived closed
forms, numpy einsum; the weight gradient against numpy einsum, the adjoint
identity with the einsum and the linearity of the fused forward in W; the
error scale S = sum |terms| returned beside every output against |M| of the
independent dense matrix and numpy einsum of absolute values).
"""
from __future__ import annotations

import ctypes
import os
import platform
import subprocess
from dataclasses import dataclass

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "disco_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB = os.path.join(_BUILD, f"liboracle_{platform.machine()}.so")

ISO, ANISO, INDICATOR = 0, 1, 2

_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (no fp contraction, OpenMP)."""
    os.makedirs(_BUILD, exist_ok=True)
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=gnu11", "-fopenmp", "-ffp-contract=off", "-fPIC",
               "-shared", "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        P = ctypes.c_void_p
        i32, i64, f64 = ctypes.c_int32, ctypes.c_int64, ctypes.c_double
        lib.oracle_colat.restype = f64
        lib.oracle_colat.argtypes = [i32, i32, i32]
        lib.oracle_quad.restype = f64
        lib.oracle_quad.argtypes = [i32, i32, i32]
        lib.oracle_gauss_node.restype = None
        lib.oracle_gauss_node.argtypes = [i32, i32, P, P]
        lib.oracle_hat.restype = f64
        lib.oracle_hat.argtypes = [f64, i32, f64]
        lib.oracle_geometry.restype = None
        lib.oracle_geometry.argtypes = [f64, f64, i32, i32, P, P]
        lib.oracle_basis_K.restype = i32
        lib.oracle_basis_K.argtypes = [i32, i32]
        grid6 = [i32] * 6
        lib.oracle_psi_count.restype = ctypes.c_int
        lib.oracle_psi_count.argtypes = grid6 + [i32, i32, f64, P, P]
        lib.oracle_psi_fill.restype = ctypes.c_int
        lib.oracle_psi_fill.argtypes = grid6 + [i32, i32, f64, P, P, P, P, P, P]
        lib.oracle_dense_matrix.restype = ctypes.c_int
        lib.oracle_dense_matrix.argtypes = grid6 + [i32, i32, f64, P]
        shape = [i32, i32, i32, i32, i32]  # K, Hin, Win, Hout, Wout
        lib.oracle_fwd.restype = None
        lib.oracle_fwd.argtypes = [P, P, P] + shape + [i64, P, P, P, P]
        lib.oracle_bwd.restype = None
        lib.oracle_bwd.argtypes = [P, P, P] + shape + [i64, P, P, P, P]
        lib.oracle_einsum.restype = None
        lib.oracle_einsum.argtypes = [P, i32, i32, i32, i64, i32, P, P, P, P]
        lib.oracle_einsum_t.restype = None
        lib.oracle_einsum_t.argtypes = [P, i32, i32, i32, i64, i32, P, P, P]
        lib.oracle_einsum_w.restype = None
        lib.oracle_einsum_w.argtypes = [P, P, P, i32, i32, i32, i64, i32, P, P]
        lib.oracle_fwd_points.restype = None
        lib.oracle_fwd_points.argtypes = [P, P, P] + shape + [P, i64, P, P, P]
        lib.oracle_bwd_points.restype = None
        lib.oracle_bwd_points.argtypes = [P, P, P] + shape + [P, i64, P, P, P]
        lib.oracle_fused_points.restype = None
        lib.oracle_fused_points.argtypes = [P, P, P] + shape + [i32, i32, P, P, i64, P, P, P]
        lib.oracle_fused_bwd_points.restype = None
        lib.oracle_fused_bwd_points.argtypes = [P, P, P] + shape + [i32, i32, P, P, i64, P, P, P]
        _lib = lib
    return _lib


def _p(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _f64(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _f32(a) -> np.ndarray:
    """fp32 storage of inputs that are exactly fp32 (or bf16) values."""
    a = np.asarray(a)
    if a.dtype != np.float32:
        b = a.astype(np.float32)
        if not np.array_equal(b.astype(a.dtype), a):
            raise ValueError("sampled oracle inputs must be exactly representable in fp32")
        a = b
    return np.ascontiguousarray(a)


# ------------------------------------------------------------------ geometry

def colat(nlat: int, poles: int, i: int) -> float:
    return _load().oracle_colat(nlat, poles, i)


def quad(nlat: int, poles: int, i: int) -> float:
    return _load().oracle_quad(nlat, poles, i)


def gauss_node(n: int, i: int):
    """(x_i, w_i): the i-th Gauss-Legendre node of order n (descending) and its weight."""
    x, w = ctypes.c_double(), ctypes.c_double()
    _load().oracle_gauss_node(n, i, ctypes.byref(x), ctypes.byref(w))
    return x.value, w.value


def hat(d: float, r: int, width: float) -> float:
    return _load().oracle_hat(d, r, width)


def geometry(th_o: float, th_i: float, delta: int, W: int):
    d = ctypes.c_double()
    b = ctypes.c_double()
    _load().oracle_geometry(th_o, th_i, delta, W, ctypes.byref(d), ctypes.byref(b))
    return d.value, b.value


def basis_K(kind: int, nrad: int) -> int:
    return _load().oracle_basis_K(kind, nrad)


# ----------------------------------------------------------------------- psi

@dataclass
class OraclePsi:
    """psi in both layouts, fp64 values.

    Union ("kpacked") layout: row_ptr[Hout+1], idx[nnz, 2] = (hi, wi),
    val[nnz, K].  CSR layout: rows k*Hout + ho, csr_col = hi*Win + wi."""
    grid_in: tuple
    grid_out: tuple
    kind: int
    nrad: int
    cutoff: float
    K: int
    row_ptr: np.ndarray
    idx: np.ndarray
    val: np.ndarray
    csr_row_ptr: np.ndarray
    csr_col: np.ndarray
    csr_val: np.ndarray

    @property
    def Hin(self):
        return self.grid_in[0]

    @property
    def Win(self):
        return self.grid_in[1]

    @property
    def Hout(self):
        return self.grid_out[0]

    @property
    def Wout(self):
        return self.grid_out[1]

    def _shape(self):
        return (self.K, self.Hin, self.Win, self.Hout, self.Wout)

    def _csr(self):
        return (_p(self.csr_row_ptr), _p(self.csr_col), _p(self.csr_val))


def build_psi(grid_in, grid_out, kind: int, nrad: int, cutoff: float) -> OraclePsi:
    """grid = (nlat, nlon, poles)."""
    lib = _load()
    gi, go = tuple(int(v) for v in grid_in), tuple(int(v) for v in grid_out)
    nnz = ctypes.c_int64()
    nnz_csr = ctypes.c_int64()
    rc = lib.oracle_psi_count(*gi, *go, kind, nrad, float(cutoff), ctypes.byref(nnz),
                              ctypes.byref(nnz_csr))
    if rc != 0:
        raise ValueError("oracle_psi_count rejected the arguments")
    K = basis_K(kind, nrad)
    Hout = go[0]
    row_ptr = np.zeros(Hout + 1, np.int64)
    idx = np.zeros((nnz.value, 2), np.int32)
    val = np.zeros((nnz.value, K), np.float64)
    csr_row_ptr = np.zeros(K * Hout + 1, np.int64)
    csr_col = np.zeros(nnz_csr.value, np.int32)
    csr_val = np.zeros(nnz_csr.value, np.float64)
    rc = lib.oracle_psi_fill(*gi, *go, kind, nrad, float(cutoff), _p(row_ptr), _p(idx), _p(val),
                             _p(csr_row_ptr), _p(csr_col), _p(csr_val))
    if rc != 0:
        raise ValueError("oracle_psi_fill rejected the arguments")
    return OraclePsi(gi, go, kind, nrad, float(cutoff), K, row_ptr, idx, val, csr_row_ptr,
                     csr_col, csr_val)


def dense_matrix(grid_in, grid_out, kind: int, nrad: int, cutoff: float) -> np.ndarray:
    """[K*Hout*Wout, Hin*Win] evaluated at the true output longitudes."""
    gi, go = tuple(int(v) for v in grid_in), tuple(int(v) for v in grid_out)
    K = basis_K(kind, nrad)
    M = np.zeros((K * go[0] * go[1], gi[0] * gi[1]), np.float64)
    if _load().oracle_dense_matrix(*gi, *go, kind, nrad, float(cutoff), _p(M)) != 0:
        raise ValueError("oracle_dense_matrix rejected the arguments")
    return M


# -------------------------------------------------------------- contractions

def fwd(psi: OraclePsi, x, xabs=None):
    """x[B, C, Hin, Win] -> (X[B, C, K, Hout, Wout], S)."""
    x = _f64(x)
    B, C = x.shape[:2]
    X = np.empty((B, C, psi.K, psi.Hout, psi.Wout), np.float64)
    S = np.empty_like(X)
    xa = _f64(xabs) if xabs is not None else None
    _load().oracle_fwd(*psi._csr(), *psi._shape(), B * C, _p(x),
                       _p(xa) if xa is not None else None, _p(X), _p(S))
    return X, S


def bwd(psi: OraclePsi, G, Gabs=None):
    """G[B, C, K, Hout, Wout] -> (gx[B, C, Hin, Win], S)."""
    G = _f64(G)
    B, C = G.shape[:2]
    gx = np.empty((B, C, psi.Hin, psi.Win), np.float64)
    S = np.empty_like(gx)
    ga = _f64(Gabs) if Gabs is not None else None
    _load().oracle_bwd(*psi._csr(), *psi._shape(), B * C, _p(G),
                       _p(ga) if ga is not None else None, _p(gx), _p(S))
    return gx, S


def einsum(W, X, SX=None):
    """W[Cout, Cin, K], X[B, Cin, K, Hout, Wout] -> (y[B, Cout, Hout, Wout], Sy)."""
    W, X = _f64(W), _f64(X)
    Cout, Cin, K = W.shape
    B = X.shape[0]
    P = X.shape[3] * X.shape[4]
    y = np.empty((B, Cout) + X.shape[3:], np.float64)
    Sy = np.empty_like(y)
    sx = _f64(SX) if SX is not None else np.abs(X)
    _load().oracle_einsum(_p(W), Cout, Cin, K, P, B, _p(X), _p(sx), _p(y), _p(Sy))
    return y, Sy


def einsum_t(W, dy):
    """W[Cout, Cin, K], dy[B, Cout, Hout, Wout] -> (dX[B, Cin, K, Hout, Wout], SdX)."""
    W, dy = _f64(W), _f64(dy)
    Cout, Cin, K = W.shape
    B = dy.shape[0]
    P = dy.shape[2] * dy.shape[3]
    dX = np.empty((B, Cin, K) + dy.shape[2:], np.float64)
    SdX = np.empty_like(dX)
    _load().oracle_einsum_t(_p(W), Cout, Cin, K, P, B, _p(dy), _p(dX), _p(SdX))
    return dX, SdX


def einsum_w(dy, X, SX=None):
    """dy[B, Cout, Hout, Wout], X[B, Cin, K, Hout, Wout] -> (dW[Cout, Cin, K], SdW):
    the weight gradient of y = einsum(W, X), dW[o,c,k] = sum_{b,p} dy[b,o,p] X[b,c,k,p]."""
    dy, X = _f64(dy), _f64(X)
    B, Cout = dy.shape[:2]
    Cin, K = X.shape[1], X.shape[2]
    P = dy.shape[2] * dy.shape[3]
    dW = np.empty((Cout, Cin, K), np.float64)
    SdW = np.empty_like(dW)
    sx = _f64(SX) if SX is not None else None
    _load().oracle_einsum_w(_p(dy), _p(X), _p(sx) if sx is not None else None, Cout, Cin, K, P, B,
                            _p(dW), _p(SdW))
    return dW, SdW


def fused_bwd_weight(psi: OraclePsi, x, dy):
    """Weight gradient of the fused forward: dW = sum_{b,p} dy * fwd(x)."""
    X, SX = fwd(psi, x)
    return einsum_w(dy, X, SX)


def fused(psi: OraclePsi, x, W):
    """Fused forward y = einsum(W, fwd(x)), with S = sum |W psi x|."""
    X, SX = fwd(psi, x)
    return einsum(W, X, SX)


def fused_bwd_input(psi: OraclePsi, dy, W):
    """Input gradient of the fused forward: gx = psi^T (W^T dy)."""
    dX, SdX = einsum_t(W, dy)
    return bwd(psi, dX, SdX)


def _pts(pts, width):
    pts = np.ascontiguousarray(np.asarray(pts, dtype=np.int64).reshape(-1, width))
    return pts, pts.shape[0]


def fwd_points(psi: OraclePsi, x, pts):
    """pts[:, 4] = (b*C + c, k, ho, wo) -> (X at those points, S)."""
    x = _f32(x)
    pts, n = _pts(pts, 4)
    out, S = np.empty(n), np.empty(n)
    _load().oracle_fwd_points(*psi._csr(), *psi._shape(), _p(x), n, _p(pts), _p(out), _p(S))
    return out, S


def bwd_points(psi: OraclePsi, G, pts):
    """pts[:, 3] = (b*C + c, hi, wi) -> (gx at those points, S)."""
    G = _f32(G)
    pts, n = _pts(pts, 3)
    out, S = np.empty(n), np.empty(n)
    _load().oracle_bwd_points(*psi._csr(), *psi._shape(), _p(G), n, _p(pts), _p(out), _p(S))
    return out, S


def fused_points(psi: OraclePsi, x, W, pts):
    """pts[:, 4] = (b, o, ho, wo) -> (y at those points, S)."""
    x, W = _f32(x), _f32(W)
    Cout, Cin, _ = W.shape
    pts, n = _pts(pts, 4)
    out, S = np.empty(n), np.empty(n)
    _load().oracle_fused_points(*psi._csr(), *psi._shape(), Cin, Cout, _p(x), _p(W), n,
                                _p(pts), _p(out), _p(S))
    return out, S


def fused_bwd_points(psi: OraclePsi, dy, W, pts):
    """pts[:, 4] = (b, c, hi, wi) -> (gx at those points, S)."""
    dy, W = _f32(dy), _f32(W)
    Cout, Cin, _ = W.shape
    pts, n = _pts(pts, 4)
    out, S = np.empty(n), np.empty(n)
    _load().oracle_fused_bwd_points(*psi._csr(), *psi._shape(), Cin, Cout, _p(dy), _p(W), n,
                                    _p(pts), _p(out), _p(S))
    return out, S
