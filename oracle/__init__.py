"""fp64 CPU oracle of the LoRA linear layer -- TEST INFRASTRUCTURE.

Only `tests/`, `__graft_entry__.smoke()` and the CPU-baseline leg of
`bench.py` may import this package.  The CUDA product path never does, and
this package imports nothing from it.

The arithmetic lives in `lora_oracle.c` (plain loops, fp64, OpenMP over
output rows).  This module only compiles it with gcc, loads it with ctypes and
converts tensors/arrays to contiguous float64 numpy arrays (an exact upcast of
bf16 or fp32 values).

Equations (ch05 "Acceleration principles: Triton kernels and fused LoRA",
§5.3; ch01 "Project background", §1.2), with s = alpha / r:
    H  = X A^T                 Y  = X W^T + s H B^T
    G  = dY B                  dX = dY W + s G A
    dA = s G^T X               dB = s dY^T H
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "lora_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liblora_oracle.so")
_lib = None
_lock = threading.Lock()

_D = ctypes.POINTER(ctypes.c_double)
_I = ctypes.POINTER(ctypes.c_int64)
_i64 = ctypes.c_int64

_SIGS = {
    "lora_oracle_threads": ([], ctypes.c_int),
    "lora_oracle_h": ([_D, _D, _i64, _i64, _i64, _D], None),
    "lora_oracle_g": ([_D, _D, _i64, _i64, _i64, _D], None),
    "lora_oracle_y": ([_D, _D, _D, _D, ctypes.c_double, _i64, _i64, _i64, _i64, _D], None),
    "lora_oracle_dx": ([_D, _D, _D, _D, ctypes.c_double, _i64, _i64, _i64, _i64, _D], None),
    "lora_oracle_da": ([_D, _D, ctypes.c_double, _i64, _i64, _i64, _D], None),
    "lora_oracle_db": ([_D, _D, ctypes.c_double, _i64, _i64, _i64, _D], None),
    "lora_oracle_h_col": ([_D, _D, _i64, _i64, _i64, _D], None),
    "lora_oracle_g_col": ([_D, _D, _i64, _i64, _i64, _i64, _D], None),
    "lora_oracle_h_rows": ([_D, _D, _i64, _i64, _I, _i64, _D], None),
    "lora_oracle_g_rows": ([_D, _D, _i64, _i64, _I, _i64, _D], None),
    "lora_oracle_y_rows": ([_D, _D, _D, _D, ctypes.c_double, _i64, _i64, _i64, _I, _i64, _D], None),
    "lora_oracle_dx_rows": ([_D, _D, _D, _D, ctypes.c_double, _i64, _i64, _i64, _I, _i64, _D], None),
    "lora_oracle_da_entries": ([_D, _D, ctypes.c_double, _i64, _i64, _I, _i64, _D], None),
    "lora_oracle_db_entries": ([_D, _D, ctypes.c_double, _i64, _i64, _I, _i64, _D], None),
}


def compile_library(src: str = _SRC, out: str = _LIB_PATH) -> str:
    """Compile the oracle with gcc into a shared library; returns its path."""
    cmd = ["gcc", "-O2", "-fopenmp", "-ffp-contract=off", "-fPIC", "-shared",
           "-std=c11", src, "-o", out]
    subprocess.run(cmd, check=True)
    return out


def load(path: str | None = None, rebuild: bool = False):
    """Load (compiling first if needed) the oracle library."""
    global _lib
    with _lock:
        if path is None and _lib is not None and not rebuild:
            return _lib
        p = path or _LIB_PATH
        if path is None and (rebuild or not os.path.exists(p)
                             or os.path.getmtime(p) < os.path.getmtime(_SRC)):
            compile_library()
        lib = ctypes.CDLL(p)
        for name, (args, res) in _SIGS.items():
            f = getattr(lib, name)
            f.argtypes = args
            f.restype = res
        if path is None:
            _lib = lib
        return lib


def _f64(a) -> np.ndarray:
    """Exact upcast of a torch tensor or array to contiguous float64."""
    try:
        import torch
        if isinstance(a, torch.Tensor):
            a = a.detach().to("cpu", torch.float64).numpy()
    except ImportError:  # pragma: no cover
        pass
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _p(a: np.ndarray):
    return a.ctypes.data_as(_D)


def _ip(a: np.ndarray):
    return a.ctypes.data_as(_I)


def _rowdot(lib, P, Q) -> np.ndarray:
    """out[a][b] = sum_k P[a][k] Q[b][k] (k ascending), by the H routine."""
    out = np.empty((P.shape[0], Q.shape[0]))
    lib.lora_oracle_h(_p(P), _p(Q), P.shape[0], P.shape[1], Q.shape[0], _p(out))
    return out


def threads(lib=None) -> int:
    return (lib or load()).lora_oracle_threads()


def scale(alpha: float, r: int) -> float:
    """s = alpha / r (ch05 §5.3 LoRA equation)."""
    return float(alpha) / float(r)


def forward(X, W, A, B, alpha: float, lib=None):
    """Returns (H, Y) as float64 arrays: H = X A^T, Y = X W^T + s H B^T."""
    lib = lib or load()
    X, W, A, B = map(_f64, (X, W, A, B))
    M, d_in = X.shape
    d_out, r = B.shape
    s = scale(alpha, r)
    H = np.empty((M, r))
    Y = np.empty((M, d_out))
    lib.lora_oracle_h(_p(X), _p(A), M, d_in, r, _p(H))
    lib.lora_oracle_y(_p(X), _p(W), _p(B), _p(H), s, M, d_in, d_out, r, _p(Y))
    return H, Y


def backward(dY, X, W, A, B, alpha: float, lib=None):
    """Returns (dX, dA, dB) as float64 arrays for the loss L = <dY, Y>."""
    lib = lib or load()
    dY, X, W, A, B = map(_f64, (dY, X, W, A, B))
    M, d_in = X.shape
    d_out, r = B.shape
    s = scale(alpha, r)
    H = np.empty((M, r))
    G = np.empty((M, r))
    dX = np.empty((M, d_in))
    dA = np.empty((r, d_in))
    dB = np.empty((d_out, r))
    lib.lora_oracle_h(_p(X), _p(A), M, d_in, r, _p(H))
    lib.lora_oracle_g(_p(dY), _p(B), M, d_out, r, _p(G))
    lib.lora_oracle_dx(_p(dY), _p(W), _p(A), _p(G), s, M, d_in, d_out, r, _p(dX))
    lib.lora_oracle_da(_p(G), _p(X), s, M, d_in, r, _p(dA))
    lib.lora_oracle_db(_p(dY), _p(H), s, M, d_out, r, _p(dB))
    return dX, dA, dB


def loss(dY, X, W, A, B, alpha: float, lib=None) -> float:
    """L = <dY, Y> computed from the oracle's forward (sum in fp64)."""
    _, Y = forward(X, W, A, B, alpha, lib=lib)
    return float(np.sum(_f64(dY) * Y))


class Sampled:
    """Oracle values for chosen rows / entries of a large problem.

    Each value is the same per-element sum as the full routines compute, so
    sampled and full results agree bit for bit.  Inputs are upcast once.
    """

    def __init__(self, X, W, A, B, dY, alpha: float, lib=None):
        self.lib = lib or load()
        self.X, self.W, self.A, self.B = map(_f64, (X, W, A, B))
        self.dY = _f64(dY) if dY is not None else None
        self.M, self.d_in = self.X.shape
        self.d_out, self.r = self.B.shape
        self.s = scale(alpha, self.r)
        self._H = None
        self._G = None

    def H(self) -> np.ndarray:
        if self._H is None:
            self._H = np.empty((self.M, self.r))
            self.lib.lora_oracle_h(_p(self.X), _p(self.A), self.M, self.d_in,
                                   self.r, _p(self._H))
        return self._H

    def G(self) -> np.ndarray:
        """G = dY B.  The H routine on (dY, B^T) forms, for every element, the
        same products in the same order (o ascending) as the G routine, so
        the bits are the same; it reads rows of B^T instead of columns of B,
        which keeps a wide B in cache."""
        if self._G is None:
            self._G = _rowdot(self.lib, self.dY, np.ascontiguousarray(self.B.T))
        return self._G

    def dA(self) -> np.ndarray:
        """All of dA = s G^T X, [r, d_in]: s times the row dot products of
        G^T and X^T (each element the sum over m ascending, then scaled, as
        the dA routine forms it)."""
        return self.s * _rowdot(self.lib, np.ascontiguousarray(self.G().T),
                                np.ascontiguousarray(self.X.T))

    def dB(self) -> np.ndarray:
        """All of dB = s dY^T H, [d_out, r], likewise from dY^T and H^T."""
        return self.s * _rowdot(self.lib, np.ascontiguousarray(self.dY.T),
                                np.ascontiguousarray(self.H().T))

    # The products with the frozen W, taken by numpy's float64 matmul (a
    # library GEMM as one step, summing in its own order): the plain loops
    # stream all of W once per output row, which takes minutes on the
    # largest shapes.  The low-rank terms come from the plain loops.
    def y_rows_mm(self, rows) -> np.ndarray:
        """Y[rows] = X[rows] W^T + s H[rows] B^T."""
        rows = np.ascontiguousarray(rows, dtype=np.int64)
        H = self._h_rows(rows)[rows]
        return self.X[rows] @ self.W.T + self.s * (H @ self.B.T)

    def dx_rows_mm(self, rows) -> np.ndarray:
        """dX[rows] = dY[rows] W + s G[rows] A."""
        rows = np.ascontiguousarray(rows, dtype=np.int64)
        G = self._g_rows(rows)[rows]
        return self.dY[rows] @ self.W + self.s * (G @ self.A)

    def _h_rows(self, rows) -> np.ndarray:
        if self._H is not None:
            return self._H
        H = np.zeros((self.M, self.r))
        self.lib.lora_oracle_h_rows(_p(self.X), _p(self.A), self.d_in, self.r,
                                    _ip(rows), len(rows), _p(H))
        return H

    def _g_rows(self, rows) -> np.ndarray:
        if self._G is not None:
            return self._G
        G = np.zeros((self.M, self.r))
        self.lib.lora_oracle_g_rows(_p(self.dY), _p(self.B), self.d_out, self.r,
                                    _ip(rows), len(rows), _p(G))
        return G

    def y_rows(self, rows) -> np.ndarray:
        rows = np.ascontiguousarray(rows, dtype=np.int64)
        out = np.empty((len(rows), self.d_out))
        H = self._h_rows(rows)
        self.lib.lora_oracle_y_rows(_p(self.X), _p(self.W), _p(self.B), _p(H),
                                    self.s, self.d_in, self.d_out, self.r,
                                    _ip(rows), len(rows), _p(out))
        return out

    def dx_rows(self, rows) -> np.ndarray:
        rows = np.ascontiguousarray(rows, dtype=np.int64)
        out = np.empty((len(rows), self.d_in))
        G = self._g_rows(rows)
        self.lib.lora_oracle_dx_rows(_p(self.dY), _p(self.W), _p(self.A), _p(G),
                                     self.s, self.d_in, self.d_out, self.r,
                                     _ip(rows), len(rows), _p(out))
        return out

    def _col(self, which: str, i: int) -> np.ndarray:
        out = np.empty(self.M)
        if which == "h":
            self.lib.lora_oracle_h_col(_p(self.X), _p(self.A), self.M, self.d_in,
                                       int(i), _p(out))
        else:
            self.lib.lora_oracle_g_col(_p(self.dY), _p(self.B), self.M,
                                       self.d_out, self.r, int(i), _p(out))
        return out

    def da_entries(self, ii, kk) -> np.ndarray:
        """dA[ii[j], kk[j]] for each j."""
        ii = np.asarray(ii, dtype=np.int64)
        kk = np.ascontiguousarray(kk, dtype=np.int64)
        cache = {}
        cols = np.empty((len(ii), self.M))
        for j, i in enumerate(ii):
            if int(i) not in cache:
                cache[int(i)] = (self.G()[:, int(i)].copy() if self._G is not None
                                 else self._col("g", int(i)))
            cols[j] = cache[int(i)]
        cols = np.ascontiguousarray(cols)
        out = np.empty(len(ii))
        self.lib.lora_oracle_da_entries(_p(cols), _p(self.X), self.s, self.M,
                                        self.d_in, _ip(kk), len(ii), _p(out))
        return out

    def db_entries(self, oo, ii) -> np.ndarray:
        """dB[oo[j], ii[j]] for each j."""
        oo = np.ascontiguousarray(oo, dtype=np.int64)
        ii = np.asarray(ii, dtype=np.int64)
        cache = {}
        cols = np.empty((len(ii), self.M))
        for j, i in enumerate(ii):
            if int(i) not in cache:
                cache[int(i)] = (self.H()[:, int(i)].copy() if self._H is not None
                                 else self._col("h", int(i)))
            cols[j] = cache[int(i)]
        cols = np.ascontiguousarray(cols)
        out = np.empty(len(ii))
        self.lib.lora_oracle_db_entries(_p(self.dY), _p(cols), self.s, self.M,
                                        self.d_out, _ip(oo), len(ii), _p(out))
        return out
