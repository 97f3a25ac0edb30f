"""fp64 CPU oracle for causal linear attention with phi(x) = elu(x) + 1, and for
its decayed variant, retention (a fixed decay per head, no feature map).

TEST INFRASTRUCTURE ONLY.  The tests, the smoke check and the benchmark's
CPU-baseline leg may import this package; the product library never does.  The
C source (``la_oracle.c``) shares no code with the CUDA path.

Every function takes numpy arrays (converted to contiguous fp64) in the layout
q, k: [B, H, N, Dk]; v, dO: [B, H, N, Dv] (any leading shape that flattens to
heads), and returns new fp64 arrays.  Which page and section each form follows
is stated beside each C function.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "la_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liblaoracle.so")
_lock = threading.Lock()
_lib = None

# -ffp-contract=off keeps the same rounding on x86 and aarch64 hosts.
CFLAGS = ["-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off"]


def build(force: bool = False, src: str = _SRC, out: str = _LIB_PATH) -> str:
    """Compile la_oracle.c with gcc into a shared library; return its path."""
    os.makedirs(os.path.dirname(out), exist_ok=True)
    if force or not os.path.exists(out) or os.path.getmtime(out) < os.path.getmtime(src):
        tmp = out + ".tmp%d" % os.getpid()
        subprocess.run(["gcc", *CFLAGS, "-o", tmp, src, "-lm"], check=True)
        os.replace(tmp, out)
    return out


_DP = ctypes.POINTER(ctypes.c_double)


def _declare(lib):
    i = ctypes.c_int
    for name in ("oracle_causal_direct", "oracle_noncausal_direct", "oracle_noncausal_assoc",
                 "oracle_causal_recurrent"):
        getattr(lib, name).argtypes = [_DP, _DP, _DP, _DP, i, i, i, i]
        getattr(lib, name).restype = None
    lib.oracle_causal_chunked.argtypes = [_DP, _DP, _DP, _DP, i, i, i, i, i]
    lib.oracle_causal_chunked.restype = None
    for name in ("oracle_causal_bwd_direct", "oracle_causal_bwd_recurrent",
                 "oracle_noncausal_bwd_direct", "oracle_noncausal_bwd_assoc"):
        getattr(lib, name).argtypes = [_DP] * 7 + [i, i, i, i]
        getattr(lib, name).restype = None
    lib.oracle_recurrent_step.argtypes = [_DP] * 6 + [i, i, i]
    lib.oracle_recurrent_step.restype = None
    for name in ("oracle_retention_direct", "oracle_retention_recurrent"):
        getattr(lib, name).argtypes = [_DP] * 5 + [i, i, i, i]
        getattr(lib, name).restype = None
    lib.oracle_retention_chunked.argtypes = [_DP] * 5 + [i, i, i, i, i]
    lib.oracle_retention_chunked.restype = None
    lib.oracle_retention_step.argtypes = [_DP] * 6 + [i, i, i]
    lib.oracle_retention_step.restype = None
    for name in ("oracle_phi", "oracle_dphi"):
        getattr(lib, name).argtypes = [_DP, _DP, ctypes.c_long]
        getattr(lib, name).restype = None
    return lib


def load_library(path: str):
    """Load an oracle build from an explicit path (used to test planted mistakes)."""
    return _declare(ctypes.CDLL(path))


def lib():
    global _lib
    with _lock:
        if _lib is None:
            _lib = load_library(build())
    return _lib


def _f64(a) -> np.ndarray:
    if hasattr(a, "detach"):  # torch tensor on the CPU
        a = a.detach().to("cpu").double().numpy()
    return np.ascontiguousarray(a, dtype=np.float64)


def _p(a: np.ndarray):
    return a.ctypes.data_as(_DP)


def _heads(q, k, v):
    q, k, v = _f64(q), _f64(k), _f64(v)
    N, Dk = q.shape[-2], q.shape[-1]
    Dv = v.shape[-1]
    if k.shape != q.shape or v.shape[:-1] != q.shape[:-1]:
        raise ValueError("shape mismatch: q %s k %s v %s" % (q.shape, k.shape, v.shape))
    BH = int(np.prod(q.shape[:-2])) if q.ndim > 2 else 1
    return q, k, v, BH, N, Dk, Dv


class Oracle:
    """Thin numpy front end over one loaded oracle build."""

    def __init__(self, library=None):
        self._l = library

    @property
    def l(self):
        return self._l if self._l is not None else lib()

    def phi(self, x):
        x = _f64(x)
        y = np.empty_like(x)
        self.l.oracle_phi(_p(x), _p(y), x.size)
        return y

    def dphi(self, x):
        x = _f64(x)
        y = np.empty_like(x)
        self.l.oracle_dphi(_p(x), _p(y), x.size)
        return y

    def _fwd(self, name, q, k, v, *extra):
        q, k, v, BH, N, Dk, Dv = _heads(q, k, v)
        o = np.empty(v.shape, dtype=np.float64)
        getattr(self.l, name)(_p(q), _p(k), _p(v), _p(o), BH, N, Dk, Dv, *extra)
        return o

    def causal_direct(self, q, k, v):
        return self._fwd("oracle_causal_direct", q, k, v)

    def causal_recurrent(self, q, k, v):
        return self._fwd("oracle_causal_recurrent", q, k, v)

    def causal_chunked(self, q, k, v, C):
        return self._fwd("oracle_causal_chunked", q, k, v, int(C))

    def noncausal_direct(self, q, k, v):
        return self._fwd("oracle_noncausal_direct", q, k, v)

    def noncausal_assoc(self, q, k, v):
        return self._fwd("oracle_noncausal_assoc", q, k, v)

    def _bwd(self, name, q, k, v, dO):
        q, k, v, BH, N, Dk, Dv = _heads(q, k, v)
        dO = _f64(dO)
        if dO.shape != v.shape:
            raise ValueError("dO shape %s != v shape %s" % (dO.shape, v.shape))
        dq, dk, dv = np.empty_like(q), np.empty_like(k), np.empty_like(v)
        getattr(self.l, name)(_p(q), _p(k), _p(v), _p(dO), _p(dq), _p(dk), _p(dv), BH, N, Dk, Dv)
        return dq, dk, dv

    def causal_bwd_direct(self, q, k, v, dO):
        return self._bwd("oracle_causal_bwd_direct", q, k, v, dO)

    def causal_bwd_recurrent(self, q, k, v, dO):
        return self._bwd("oracle_causal_bwd_recurrent", q, k, v, dO)

    def noncausal_bwd_direct(self, q, k, v, dO):
        return self._bwd("oracle_noncausal_bwd_direct", q, k, v, dO)

    def noncausal_bwd_assoc(self, q, k, v, dO):
        return self._bwd("oracle_noncausal_bwd_assoc", q, k, v, dO)

    # ---- retention (decay gamma per head, no feature map, no normaliser)
    @staticmethod
    def _gamma(gamma, BH):
        """gamma per flat head: given per head of one batch row ([H], tiled over B) or per flat head."""
        g = np.atleast_1d(_f64(gamma)).ravel()
        if g.size != BH and (g.size == 0 or BH % g.size != 0):
            raise ValueError("gamma has %d entries for %d heads" % (g.size, BH))
        return np.ascontiguousarray(np.tile(g, BH // g.size))

    def _ret(self, name, q, k, v, gamma, *extra):
        q, k, v, BH, N, Dk, Dv = _heads(q, k, v)
        g = self._gamma(gamma, BH)
        o = np.empty(v.shape, dtype=np.float64)
        getattr(self.l, name)(_p(q), _p(k), _p(v), _p(g), _p(o), BH, N, Dk, Dv, *extra)
        return o

    def retention_direct(self, q, k, v, gamma):
        return self._ret("oracle_retention_direct", q, k, v, gamma)

    def retention_recurrent(self, q, k, v, gamma):
        return self._ret("oracle_retention_recurrent", q, k, v, gamma)

    def retention_chunked(self, q, k, v, gamma, C):
        return self._ret("oracle_retention_chunked", q, k, v, gamma, int(C))

    def retention_step(self, q, k, v, gamma, S):
        """One retention decode step; returns (out, S') without touching the inputs."""
        q, k, v = _f64(q), _f64(k), _f64(v)
        S = _f64(S).copy()
        Dk, Dv = q.shape[-1], v.shape[-1]
        BH = q.size // Dk
        if S.size != BH * Dk * Dv or v.size != BH * Dv:
            raise ValueError("state shape mismatch")
        g = self._gamma(gamma, BH)
        out = np.empty(v.shape, dtype=np.float64)
        self.l.oracle_retention_step(_p(q), _p(k), _p(v), _p(g), _p(S), _p(out), BH, Dk, Dv)
        return out, S

    def recurrent_step(self, q, k, v, S, z):
        """One decode step; returns (out, S', z') without touching the inputs."""
        q, k, v = _f64(q), _f64(k), _f64(v)
        S, z = _f64(S).copy(), _f64(z).copy()
        Dk, Dv = q.shape[-1], v.shape[-1]
        BH = q.size // Dk
        if S.size != BH * Dk * Dv or z.size != BH * Dk or v.size != BH * Dv:
            raise ValueError("state shape mismatch")
        out = np.empty(v.shape, dtype=np.float64)
        self.l.oracle_recurrent_step(_p(q), _p(k), _p(v), _p(S), _p(z), _p(out), BH, Dk, Dv)
        return out, S, z


default = Oracle()
phi = default.phi
dphi = default.dphi
causal_direct = default.causal_direct
causal_recurrent = default.causal_recurrent
causal_chunked = default.causal_chunked
noncausal_direct = default.noncausal_direct
noncausal_assoc = default.noncausal_assoc
causal_bwd_direct = default.causal_bwd_direct
causal_bwd_recurrent = default.causal_bwd_recurrent
noncausal_bwd_direct = default.noncausal_bwd_direct
noncausal_bwd_assoc = default.noncausal_bwd_assoc
recurrent_step = default.recurrent_step
retention_direct = default.retention_direct
retention_recurrent = default.retention_recurrent
retention_chunked = default.retention_chunked
retention_step = default.retention_step
