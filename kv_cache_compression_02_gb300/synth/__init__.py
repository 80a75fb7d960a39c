"""Seeded synthetic KV-cache inputs (fp16, [L,2,H,S,d]).

The generator is plain host C (``kvgen.c``) built on demand with gcc.  It
holds none of the codec's arithmetic; it only makes the inputs that the GPU
path and the CPU oracle's tests both consume.  The recipe: per channel an
AR(1) process over tokens, ``z_t = rho z_{t-1} + sqrt(1-rho^2) e_t``, with
unit-variance Laplace or Student-t(3) innovations, scaled by lognormal(0,1)
per channel, with a few outlier channels per (layer, K/V) tensor scaled up,
rounded to fp16 after clamping to +-65504.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from dataclasses import dataclass

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kvgen.c")
_LIB = os.path.join(_HERE, "_build", "libkvgen.so")


def build(force: bool = False) -> str:
    os.makedirs(os.path.dirname(_LIB), exist_ok=True)
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".{os.getpid()}.tmp"
        subprocess.check_call(["gcc", "-O2", "-std=gnu11", "-fPIC", "-shared", "-pthread",
                               "-Wall", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


class _Spec(ctypes.Structure):
    _fields_ = [("L", ctypes.c_int32), ("H", ctypes.c_int32), ("d", ctypes.c_int32),
                ("innov", ctypes.c_int32), ("S", ctypes.c_int64), ("seed", ctypes.c_uint64),
                ("rho_lo", ctypes.c_double), ("rho_hi", ctypes.c_double),
                ("outlier_frac", ctypes.c_double), ("outlier_scale", ctypes.c_double),
                ("n_outliers", ctypes.c_int32), ("pad_", ctypes.c_int32)]


_lib = None


def _l():
    global _lib
    if _lib is None:
        _lib = ctypes.CDLL(build())
        P = ctypes.c_void_p
        _lib.kvgen_head.argtypes = [P, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, P]
        _lib.kvgen_head.restype = None
        _lib.kvgen_range.argtypes = [P, ctypes.c_int64, ctypes.c_int64, P, ctypes.c_int32]
        _lib.kvgen_range.restype = None
        _lib.kvgen_channel.argtypes = [P, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, P, P]
        _lib.kvgen_channel.restype = None
        _lib.kvgen_chunk_levels.argtypes = [ctypes.c_uint64, ctypes.c_int64, ctypes.c_int32, P]
        _lib.kvgen_chunk_levels.restype = None
    return _lib


@dataclass(frozen=True)
class GenSpec:
    L: int
    H: int
    d: int
    S: int
    seed: int
    innov: str = "laplace"          # "laplace" or "t3"
    rho: tuple = (0.95, 0.95)       # fixed, or U(lo, hi) per channel
    outlier_frac: float = 0.0
    outlier_scale: float = 10.0
    n_outliers: int = -1            # exact count per tensor when >= 0

    def _c(self) -> _Spec:
        return _Spec(self.L, self.H, self.d, 1 if self.innov == "t3" else 0, self.S,
                     self.seed & (2**64 - 1), self.rho[0], self.rho[1], self.outlier_frac,
                     self.outlier_scale, self.n_outliers, 0)

    @property
    def n_heads(self) -> int:
        return self.L * 2 * self.H

    @property
    def shape(self):
        return (self.L, 2, self.H, self.S, self.d)


def threads() -> int:
    return max(1, os.cpu_count() or 1)


def head(spec: GenSpec, l: int, kv: int, h: int) -> np.ndarray:
    """One head's [S][d] fp16 bits (uint16)."""
    out = np.empty((spec.S, spec.d), np.uint16)
    sp = spec._c()
    _l().kvgen_head(ctypes.byref(sp), l, kv, h, out.ctypes.data_as(ctypes.c_void_p))
    return out


def fill(spec: GenSpec, ptr: int, h0: int = 0, h1: int | None = None, nthreads: int | None = None):
    """Write heads [h0, h1) (flattened (l,kv,h) order) to host memory at ptr."""
    h1 = spec.n_heads if h1 is None else h1
    sp = spec._c()
    _l().kvgen_range(ctypes.byref(sp), h0, h1, ctypes.c_void_p(ptr), nthreads or threads())


def generate(spec: GenSpec, nthreads: int | None = None) -> np.ndarray:
    out = np.empty(spec.shape, np.uint16)
    fill(spec, out.ctypes.data, nthreads=nthreads)
    return out


def channel(spec: GenSpec, l: int, kv: int, c: int):
    rho, sc = ctypes.c_double(), ctypes.c_double()
    sp = spec._c()
    _l().kvgen_channel(ctypes.byref(sp), l, kv, c, ctypes.byref(rho), ctypes.byref(sc))
    return rho.value, sc.value


def chunk_levels(seed: int, n_chunks: int, n_levels: int) -> np.ndarray:
    out = np.empty(n_chunks, np.uint8)
    _l().kvgen_chunk_levels(seed & (2**64 - 1), n_chunks, n_levels, out.ctypes.data_as(ctypes.c_void_p))
    return out
