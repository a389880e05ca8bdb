"""Python face of the plain C++ oracle (``oracle/lynx_oracle.cpp``).

TEST INFRASTRUCTURE.  Only the tests, ``__graft_entry__.smoke()`` and the CPU
arms of ``bench.py`` may import or run this module; the library never does.

The functions have the names and arguments of the numpy oracle
(``oracle/lynx_oracle.py``), so that one pin suite checks both.  Inputs are
uint16 arrays of bf16 bit patterns, row-major; results are float64.  Each call
splits its rows over ``threads`` std::threads (default: every host core, or
``LYNX_ORACLE_THREADS``); the result does not depend on the thread count.

``build()`` compiles the C++ file with the host compiler (plain ``g++``, no
machine-specific flags) into ``oracle/liblynx_oracle.so``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(HERE, "lynx_oracle.cpp")
LIB = os.path.join(HERE, "liblynx_oracle.so")

__all__ = ["build", "CppOracle", "default", "widen", "select_2of4", "keep_mask", "norm_scale", "canonical_meta",
           "sparsify", "linear", "lora_down", "linear_dense", "linear_wsparse", "round_bf16", "gelu", "gelu_bf16",
           "mlp_input", "NIBBLE_OF_PAIR", "host_threads"]

#: 4-bit metadata of a kept index pair (i0 < i1): i0 in bits 0-1, i1 in bits 2-3.
NIBBLE_OF_PAIR = {(i0, i1): i0 | (i1 << 2) for i0 in range(4) for i1 in range(i0 + 1, 4)}


def build(source: str = SOURCE, out: str = LIB, force: bool = False) -> str:
    """Compile the oracle into a shared library (only when the source is newer than the library)."""
    if not force and os.path.exists(out) and os.path.getmtime(out) >= os.path.getmtime(source):
        return out
    cxx = os.environ.get("CXX", "g++")
    tmp = f"{out}.{os.getpid()}.tmp"
    cmd = [cxx, "-O2", "-std=c++17", "-fPIC", "-shared", "-pthread", source, "-o", tmp]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"building the C++ oracle failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, out)
    return out


def host_threads() -> int:
    env = os.environ.get("LYNX_ORACLE_THREADS")
    if env and env.isdigit() and int(env) > 0:
        return int(env)
    return os.cpu_count() or 1


_u16p = ctypes.POINTER(ctypes.c_uint16)
_u8p = ctypes.POINTER(ctypes.c_uint8)
_i32p = ctypes.POINTER(ctypes.c_int32)
_i64p = ctypes.POINTER(ctypes.c_int64)
_f64p = ctypes.POINTER(ctypes.c_double)
_i64 = ctypes.c_int64


def _p(a: np.ndarray | None, ctype):
    return None if a is None else a.ctypes.data_as(ctype)


def _bits(a) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.uint16)


class CppOracle:
    """The oracle functions bound to one build of the C++ library (the default build, or a variant)."""

    def __init__(self, path: str | None = None):
        if path is None:
            path = build()
        L = ctypes.CDLL(path)
        sig = {
            "lo_version": (ctypes.c_int, []),
            "lo_widen": (None, [_u16p, _i64, _f64p]),
            "lo_select_2of4": (ctypes.c_int, [_f64p, _i64, _i64, _i32p, _i32p, ctypes.c_int]),
            "lo_keep_mask": (ctypes.c_int, [_f64p, _i64, _i64, _u8p, ctypes.c_int]),
            "lo_norm_scale": (ctypes.c_int, [_f64p, _u8p, _i64, _i64, _f64p, ctypes.c_int]),
            "lo_canonical_meta": (ctypes.c_int, [_i32p, _i32p, _i64, _i64, _u8p]),
            "lo_sparsify": (ctypes.c_int, [_u16p, _i64, _i64, _u8p, _u16p, _u8p, _f64p, ctypes.c_int]),
            "lo_linear": (ctypes.c_int, [_u16p, _u16p, _u16p, _u16p, _i64, _i64, _i64, _i64, _i64p, _i64, _f64p,
                                         ctypes.c_int]),
            "lo_lora_down": (ctypes.c_int, [_u16p, _u16p, _f64p, _i64, _i64, _i64, _f64p, ctypes.c_int]),
            "lo_linear_dense": (ctypes.c_int, [_u16p, _u16p, _u16p, _u16p, _i64, _i64, _i64, _i64, _i64p, _i64,
                                               _f64p, ctypes.c_int]),
            "lo_linear_wsparse": (ctypes.c_int, [_u16p, _u16p, _u16p, _u16p, _i64, _i64, _i64, _i64, _i64p, _i64,
                                                 _f64p, ctypes.c_int]),
            "lo_round_bf16": (None, [_f64p, _i64, _u16p]),
            "lo_gelu": (None, [_f64p, _i64, _f64p]),
            "lo_gelu_bf16": (None, [_u16p, _i64, _u16p]),
        }
        for name, (res, args) in sig.items():
            f = getattr(L, name)
            f.restype, f.argtypes = res, args
        self.lib = L
        self.path = path
        self.threads = host_threads()
        self.NIBBLE_OF_PAIR = NIBBLE_OF_PAIR

    @staticmethod
    def _ok(status: int, where: str) -> None:
        if status != 0:
            raise ValueError(f"{where}: bad shape (status {status})")

    # ---------------------------------------------------------------- element-level functions
    def widen(self, bits) -> np.ndarray:
        b = _bits(bits)
        out = np.empty(b.shape, dtype=np.float64)
        self.lib.lo_widen(_p(b, _u16p), b.size, _p(out, _f64p))
        return out

    def select_2of4(self, x) -> tuple[np.ndarray, np.ndarray]:
        x = np.ascontiguousarray(x, dtype=np.float64)
        M, K = x.shape
        if K % 4:
            raise ValueError("K must be a multiple of 4")
        i0 = np.empty((M, K // 4), dtype=np.int32)
        i1 = np.empty((M, K // 4), dtype=np.int32)
        self._ok(self.lib.lo_select_2of4(_p(x, _f64p), M, K, _p(i0, _i32p), _p(i1, _i32p), self.threads),
                 "select_2of4")
        return i0, i1

    def keep_mask(self, x) -> np.ndarray:
        x = np.ascontiguousarray(x, dtype=np.float64)
        M, K = x.shape
        keep = np.empty((M, K), dtype=np.uint8)
        self._ok(self.lib.lo_keep_mask(_p(x, _f64p), M, K, _p(keep, _u8p), self.threads), "keep_mask")
        return keep.astype(bool)

    def norm_scale(self, x, mask) -> np.ndarray:
        x = np.ascontiguousarray(x, dtype=np.float64)
        keep = np.ascontiguousarray(mask, dtype=np.uint8)
        M, K = x.shape
        s = np.empty(M, dtype=np.float64)
        self._ok(self.lib.lo_norm_scale(_p(x, _f64p), _p(keep, _u8p), M, K, _p(s, _f64p), self.threads),
                 "norm_scale")
        return s

    def canonical_meta(self, i0, i1) -> np.ndarray:
        a = np.ascontiguousarray(i0, dtype=np.int32)
        b = np.ascontiguousarray(i1, dtype=np.int32)
        M, G = a.shape
        if G % 2:
            raise ValueError("K must be a multiple of 8 for byte-packed metadata")
        out = np.empty((M, G // 2), dtype=np.uint8)
        self._ok(self.lib.lo_canonical_meta(_p(a, _i32p), _p(b, _i32p), M, G, _p(out, _u8p)), "canonical_meta")
        return out

    # ---------------------------------------------------------------- layer-level functions
    def sparsify(self, X) -> dict:
        Xb = _bits(X)
        M, K = Xb.shape
        keep = np.empty((M, K), dtype=np.uint8)
        vals = np.empty((M, K // 2), dtype=np.uint16)
        meta = np.empty((M, K // 8), dtype=np.uint8) if K % 8 == 0 else None
        s = np.empty(M, dtype=np.float64)
        self._ok(self.lib.lo_sparsify(_p(Xb, _u16p), M, K, _p(keep, _u8p), _p(vals, _u16p), _p(meta, _u8p),
                                      _p(s, _f64p), self.threads), "sparsify")
        return {"mask": keep.astype(bool), "vals": vals, "meta": meta, "s": s}

    def _rows(self, rows, M):
        if rows is None:
            return None, M
        r = np.ascontiguousarray(rows, dtype=np.int64)
        if r.size and (r.min() < 0 or r.max() >= M):
            raise IndexError("row index out of range")
        return r, r.size

    def linear(self, X, W, LA, LB, rows=None) -> np.ndarray:
        Xb, Wb, LAb, LBb = _bits(X), _bits(W), _bits(LA), _bits(LB)
        M, K = Xb.shape
        N, R = Wb.shape[0], LBb.shape[0]
        r, n = self._rows(rows, M)
        Y = np.empty((n, N), dtype=np.float64)
        self._ok(self.lib.lo_linear(_p(Xb, _u16p), _p(Wb, _u16p), _p(LAb, _u16p), _p(LBb, _u16p), M, N, K, R,
                                    _p(r, _i64p), n, _p(Y, _f64p), self.threads), "linear")
        return Y

    def lora_down(self, X, LB, s=None) -> np.ndarray:
        Xb, LBb = _bits(X), _bits(LB)
        M, K = Xb.shape
        R = LBb.shape[0]
        sd = None if s is None else np.ascontiguousarray(s, dtype=np.float64)
        T = np.empty((M, R), dtype=np.float64)
        self._ok(self.lib.lo_lora_down(_p(Xb, _u16p), _p(LBb, _u16p), _p(sd, _f64p), M, K, R, _p(T, _f64p),
                                       self.threads), "lora_down")
        return T

    def _dense_like(self, fn, X, W, LA, LB, rows):
        Xb, Wb = _bits(X), _bits(W)
        if (LA is None) != (LB is None):
            raise ValueError("LA and LB are both given or both None")
        LAb = None if LA is None else _bits(LA)
        LBb = None if LB is None else _bits(LB)
        M, K = Xb.shape
        N = Wb.shape[0]
        R = 0 if LBb is None else LBb.shape[0]
        r, n = self._rows(rows, M)
        Y = np.empty((n, N), dtype=np.float64)
        self._ok(fn(_p(Xb, _u16p), _p(Wb, _u16p), _p(LAb, _u16p), _p(LBb, _u16p), M, N, K, R, _p(r, _i64p), n,
                    _p(Y, _f64p), self.threads), "linear")
        return Y

    def round_bf16(self, x) -> np.ndarray:
        """Nearest bf16 (ties to even) of float64 values, as uint16 bit patterns."""
        xd = np.ascontiguousarray(x, dtype=np.float64)
        out = np.empty(xd.shape, dtype=np.uint16)
        self.lib.lo_round_bf16(_p(xd, _f64p), xd.size, _p(out, _u16p))
        return out

    def gelu(self, x) -> np.ndarray:
        """Exact-erf GELU in float64."""
        xd = np.ascontiguousarray(x, dtype=np.float64)
        out = np.empty(xd.shape, dtype=np.float64)
        self.lib.lo_gelu(_p(xd, _f64p), xd.size, _p(out, _f64p))
        return out

    def gelu_bf16(self, Y) -> np.ndarray:
        """H = bf16(GELU(Y)) of a bf16 tensor Y (bit patterns in and out)."""
        Yb = _bits(Y)
        out = np.empty(Yb.shape, dtype=np.uint16)
        self.lib.lo_gelu_bf16(_p(Yb, _u16p), Yb.size, _p(out, _u16p))
        return out

    def mlp_input(self, X, W, LA=None, LB=None, sparse=True, rows=None) -> np.ndarray:
        """The MLP down layer's input for the given rows: H = bf16(GELU(bf16(Y_up))), Y_up the up layer
        (sparse: linear, else linear_dense) in double, rounded to the up layer's bf16 output first."""
        y = self.linear(X, W, LA, LB, rows) if sparse else self.linear_dense(X, W, LA, LB, rows)
        return self.gelu_bf16(self.round_bf16(y))

    def linear_dense(self, X, W, LA=None, LB=None, rows=None) -> np.ndarray:
        return self._dense_like(self.lib.lo_linear_dense, X, W, LA, LB, rows)

    def linear_wsparse(self, X, W, LA=None, LB=None, rows=None) -> np.ndarray:
        return self._dense_like(self.lib.lo_linear_wsparse, X, W, LA, LB, rows)


_DEFAULT: CppOracle | None = None


def default() -> CppOracle:
    """The oracle bound to the default build (built on first use)."""
    global _DEFAULT
    if _DEFAULT is None:
        _DEFAULT = CppOracle()
    return _DEFAULT


def widen(bits):
    return default().widen(bits)


def select_2of4(x):
    return default().select_2of4(x)


def keep_mask(x):
    return default().keep_mask(x)


def norm_scale(x, mask):
    return default().norm_scale(x, mask)


def canonical_meta(i0, i1):
    return default().canonical_meta(i0, i1)


def sparsify(X):
    return default().sparsify(X)


def linear(X, W, LA, LB, rows=None):
    return default().linear(X, W, LA, LB, rows)


def lora_down(X, LB, s=None):
    return default().lora_down(X, LB, s)


def linear_dense(X, W, LA=None, LB=None, rows=None):
    return default().linear_dense(X, W, LA, LB, rows)


def round_bf16(x):
    return default().round_bf16(x)


def gelu(x):
    return default().gelu(x)


def gelu_bf16(Y):
    return default().gelu_bf16(Y)


def mlp_input(X, W, LA=None, LB=None, sparse=True, rows=None):
    return default().mlp_input(X, W, LA, LB, sparse, rows)


def linear_wsparse(X, W, LA=None, LB=None, rows=None):
    return default().linear_wsparse(X, W, LA, LB, rows)
