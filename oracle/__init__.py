"""fp64 CPU oracle for the fused attention forward pass (ctypes wrapper).

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
bench's CPU-baseline leg (including ``bench.py --impl reference``) may import
this package.  The product path (``attention_fa_fwd_gb300``) never imports it,
and this package never imports the product path: they share nothing but the
seeded input generators of ``fa_inputs``.

The arithmetic lives in ``attn_oracle.c`` (plain C, IEEE double, OpenMP over
heads or rows), which cites the page passage each function follows.  Inputs
are float64 numpy arrays of shape [B, H, S, D] (the exact widening of the
16-bit inputs); outputs are float64 O [B, H, S, D] and LSE [B, H, S] in
natural log.

Parity status: every function here is pinned in ``tests/test_oracle.py`` by
closed forms, invariants, brute force and an independent library routine; none
is "parity unpinned".
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import tempfile

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "attn_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB = os.path.join(_BUILD, "liboracle.so")

_I64 = ctypes.c_int64
_DP = ctypes.POINTER(ctypes.c_double)
_LP = ctypes.POINTER(ctypes.c_int64)


def build(force: bool = False, src: str = _SRC, out: str = _LIB) -> str:
    """Compile the C oracle with gcc (IEEE double, no fast-math) if needed."""
    if (not force and os.path.exists(out)
            and os.path.getmtime(out) >= os.path.getmtime(src)):
        return out
    os.makedirs(os.path.dirname(out), exist_ok=True)
    fd, tmp = tempfile.mkstemp(suffix=".so", dir=os.path.dirname(out))
    os.close(fd)
    cmd = ["gcc", "-O2", "-std=c11", "-D_GNU_SOURCE", "-fopenmp", "-fPIC", "-shared",
           "-fno-fast-math", "-ffp-contract=off", src, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def _f64(x) -> np.ndarray:
    a = np.ascontiguousarray(x, dtype=np.float64)
    if a.ndim != 4:
        raise ValueError("expected a [B, H, S, D] array")
    return a


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(_DP)


def _check(q, k, v):
    q, k, v = _f64(q), _f64(k), _f64(v)
    if not (q.shape == k.shape == v.shape):
        raise ValueError("q, k, v must share one [B, H, S, D] shape")
    return q, k, v


_ROUND = {None: 0, "fp16": 1, "bf16": 2}


class Oracle:
    """The oracle's entry points, bound to one compiled copy of the C file."""

    def __init__(self, libpath: str):
        lib = ctypes.CDLL(libpath)
        common = [_DP, _DP, _DP, _I64, _I64, _I64, ctypes.c_int, ctypes.c_double]
        lib.fa_oracle_attention.argtypes = common + [_DP, _DP, ctypes.c_int]
        lib.fa_oracle_attention_rows.argtypes = common + [_I64, _LP, _LP, _DP, _DP, ctypes.c_int]
        lib.fa_oracle_online.argtypes = common + [_I64, _DP, _DP, ctypes.c_int]
        lib.fa_oracle_lazy.argtypes = common + [_I64, ctypes.c_double, ctypes.c_int,
                                                _DP, _DP, _DP, ctypes.c_int]
        for f in ("fa_oracle_attention", "fa_oracle_attention_rows", "fa_oracle_online",
                  "fa_oracle_lazy", "fa_oracle_max_threads"):
            getattr(lib, f).restype = ctypes.c_int
        for f in ("fa_oracle_round_f16", "fa_oracle_round_bf16"):
            getattr(lib, f).argtypes = [ctypes.c_double]
            getattr(lib, f).restype = ctypes.c_double
        self.lib = lib
        self.path = libpath

    def max_threads(self) -> int:
        return self.lib.fa_oracle_max_threads()

    def attention(self, q, k, v, causal: bool, scale: float, nthreads: int = 0):
        """The definition, with each head's full S x S score matrix materialised."""
        q, k, v = _check(q, k, v)
        B, H, S, D = q.shape
        o = np.empty_like(q)
        lse = np.empty((B, H, S), dtype=np.float64)
        rc = self.lib.fa_oracle_attention(_ptr(q), _ptr(k), _ptr(v), B * H, S, D, int(causal),
                                          float(scale), _ptr(o), _ptr(lse), int(nthreads))
        if rc:
            raise RuntimeError(f"fa_oracle_attention failed ({rc})")
        return o, lse

    def attention_rows(self, q, k, v, causal: bool, scale: float, heads, rows,
                       nthreads: int = 0):
        """The definition for sampled rows; heads are flat b*H + h indices."""
        q, k, v = _check(q, k, v)
        B, H, S, D = q.shape
        heads = np.ascontiguousarray(heads, dtype=np.int64)
        rows = np.ascontiguousarray(rows, dtype=np.int64)
        if heads.shape != rows.shape or heads.ndim != 1:
            raise ValueError("heads and rows must be 1-D and of equal length")
        n = heads.shape[0]
        o = np.empty((n, D), dtype=np.float64)
        lse = np.empty((n,), dtype=np.float64)
        rc = self.lib.fa_oracle_attention_rows(_ptr(q), _ptr(k), _ptr(v), B * H, S, D,
                                               int(causal), float(scale), n,
                                               heads.ctypes.data_as(_LP),
                                               rows.ctypes.data_as(_LP), _ptr(o), _ptr(lse),
                                               int(nthreads))
        if rc:
            raise RuntimeError(f"fa_oracle_attention_rows failed ({rc})")
        return o, lse

    def attention_online(self, q, k, v, causal: bool, scale: float, tile: int,
                         nthreads: int = 0):
        """Textbook online softmax (running m, l; deferred normalisation)."""
        q, k, v = _check(q, k, v)
        B, H, S, D = q.shape
        o = np.empty_like(q)
        lse = np.empty((B, H, S), dtype=np.float64)
        rc = self.lib.fa_oracle_online(_ptr(q), _ptr(k), _ptr(v), B * H, S, D, int(causal),
                                       float(scale), int(tile), _ptr(o), _ptr(lse),
                                       int(nthreads))
        if rc:
            raise RuntimeError(f"fa_oracle_online failed ({rc})")
        return o, lse

    def attention_lazy(self, q, k, v, causal: bool, scale: float, tile: int = 128,
                       threshold: float = 8.0, p_round=None, nthreads: int = 0):
        """Base-2 lazy-rescale recurrence.  Returns (o, lse, stats); stats holds
        ``rebases`` (re-bases after a row's first tile), ``p_max`` and ``steps``."""
        q, k, v = _check(q, k, v)
        B, H, S, D = q.shape
        o = np.empty_like(q)
        lse = np.empty((B, H, S), dtype=np.float64)
        st = np.zeros(3, dtype=np.float64)
        rc = self.lib.fa_oracle_lazy(_ptr(q), _ptr(k), _ptr(v), B * H, S, D, int(causal),
                                     float(scale), int(tile), float(threshold),
                                     _ROUND[p_round], _ptr(o), _ptr(lse), _ptr(st),
                                     int(nthreads))
        if rc:
            raise RuntimeError(f"fa_oracle_lazy failed ({rc})")
        return o, lse, {"rebases": int(st[0]), "p_max": float(st[1]), "steps": int(st[2])}

    def round_f16(self, x: float) -> float:
        return self.lib.fa_oracle_round_f16(float(x))

    def round_bf16(self, x: float) -> float:
        return self.lib.fa_oracle_round_bf16(float(x))


_default = None


def default() -> Oracle:
    global _default
    if _default is None:
        _default = Oracle(build())
    return _default


def max_threads() -> int:
    return default().max_threads()


def attention(q, k, v, causal: bool, scale: float, nthreads: int = 0):
    return default().attention(q, k, v, causal, scale, nthreads)


def attention_rows(q, k, v, causal: bool, scale: float, heads, rows, nthreads: int = 0):
    return default().attention_rows(q, k, v, causal, scale, heads, rows, nthreads)


def attention_online(q, k, v, causal: bool, scale: float, tile: int, nthreads: int = 0):
    return default().attention_online(q, k, v, causal, scale, tile, nthreads)


def attention_lazy(q, k, v, causal: bool, scale: float, tile: int = 128, threshold: float = 8.0,
                   p_round=None, nthreads: int = 0):
    return default().attention_lazy(q, k, v, causal, scale, tile, threshold, p_round, nthreads)


def round_f16(x: float) -> float:
    return default().round_f16(x)


def round_bf16(x: float) -> float:
    return default().round_bf16(x)
