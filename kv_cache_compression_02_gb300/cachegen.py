"""ctypes binding of libcachegen.so (include/cachegen.h), same names as the C ABI.

Argument marshalling only: every step of fit, encode and decode runs in the
library's CUDA kernels.  Device buffers are torch tensors (their data_ptr()
is passed); streams are torch.cuda.Stream objects or None (the current
stream).  If the library has not been built the first call raises; there is
no CPU fallback.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

from . import build as _build

CG_OK, CG_ERR_INVALID_ARG, CG_ERR_NONFINITE, CG_ERR_CAPACITY, CG_ERR_CORRUPT, CG_ERR_CUDA, CG_ERR_TIMEOUT = range(7)
CG_OP_FIT, CG_OP_ENCODE, CG_OP_DECODE, CG_OP_ASSEMBLE = 0, 1, 2, 3


class cg_dims(ctypes.Structure):
    _fields_ = [("L", ctypes.c_int32), ("H", ctypes.c_int32), ("d", ctypes.c_int32), ("C", ctypes.c_int32),
                ("G", ctypes.c_int32), ("reserved", ctypes.c_int32), ("S", ctypes.c_int64)]


class cg_params(ctypes.Structure):
    _fields_ = [("n_levels", ctypes.c_int32), ("level_base", ctypes.c_float * 8),
                ("layer_mult", ctypes.c_void_p), ("alphabet_radius", ctypes.c_int32)]


class CacheGenError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"{what}: {cg_status_str(status)}")
        self.status = status


_lib = None


def lib() -> ctypes.CDLL:
    """Load libcachegen.so from the package's _build directory."""
    global _lib
    if _lib is None:
        if not os.path.exists(_build.LIB):
            raise RuntimeError(f"libcachegen.so is not built ({_build.LIB}); "
                               "run `python -c 'import __graft_entry__ as g; g.build()'`")
        L = ctypes.CDLL(_build.LIB)
        P, S = ctypes.c_void_p, ctypes.c_size_t
        D, Pr = ctypes.POINTER(cg_dims), ctypes.POINTER(cg_params)
        sig = {
            "cg_version": (ctypes.c_int32, []),
            "cg_status_str": (ctypes.c_char_p, [ctypes.c_int]),
            "cg_tables_bytes": (S, [D, Pr]),
            "cg_workspace_bytes": (S, [D, Pr, ctypes.c_int]),
            "cg_encode_bound": (ctypes.c_int, [D, Pr, ctypes.POINTER(ctypes.c_uint64)]),
            "cg_fit_tables": (ctypes.c_int, [D, Pr, P, P, P, S, P]),
            "cg_encode": (ctypes.c_int, [D, Pr, P, P, P, P, ctypes.c_uint64, P, P, S, P]),
            "cg_decode": (ctypes.c_int, [D, Pr, P, P, ctypes.c_uint64, ctypes.c_int32, ctypes.c_int32,
                                         P, P, S, P]),
            "cg_read_status": (ctypes.c_int, [P]),
            "cg_entropy_bound": (ctypes.c_int, [D, Pr, P, ctypes.c_int32, ctypes.POINTER(ctypes.c_double)]),
            "cg_host_mapped": (ctypes.c_int, [P, ctypes.POINTER(ctypes.c_void_p)]),
            "cg_decode_noalloc": (ctypes.c_int, [D, Pr, P, P, ctypes.c_uint64, ctypes.c_int32, ctypes.c_int32,
                                                 P, P, ctypes.POINTER(ctypes.c_void_p)]),
            "cg_assemble": (ctypes.c_int, [D, Pr, P, P, P, P, ctypes.c_uint64, P, P, S, P]),
            "cg_plan_levels": (ctypes.c_int, [ctypes.c_int32, ctypes.c_int32, P, P, ctypes.c_int32, ctypes.c_double,
                                              ctypes.c_double, P, P, P, ctypes.POINTER(ctypes.c_double)]),
            "cg_simulate_stream": (ctypes.c_int, [ctypes.c_int32, ctypes.c_int32, P, P, ctypes.c_int32, P, P, P,
                                                  ctypes.POINTER(ctypes.c_double)]),
            "cg_decode_layers": (ctypes.c_int, [D, Pr, P, P, ctypes.c_uint64, ctypes.c_int32, ctypes.c_int32,
                                                ctypes.c_int32, ctypes.c_int32, P, P, S, P]),
            "cg_decode_paged": (ctypes.c_int, [D, Pr, P, P, ctypes.c_uint64, ctypes.c_int32, ctypes.c_int32,
                                               P, P, ctypes.c_int32, ctypes.c_int32, P, S, P]),
        }
        for name, (res, args) in sig.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


def _ptr(t) -> int:
    if t is None:
        return 0
    if isinstance(t, int):
        return t
    return int(t.data_ptr())


def _stream(s) -> int | None:
    if s is None:
        import torch
        return torch.cuda.current_stream().cuda_stream or None
    return getattr(s, "cuda_stream", s) or None


class Config:
    """(cg_dims, cg_params) for one codec configuration; keeps the layer
    multiplier array alive for as long as the params point at it."""

    def __init__(self, L, H, d, S, C, G=10, R=127, level_base=(0.1,), layer_mult=None):
        self.dims = cg_dims(L, H, d, C, G, 0, S)
        self._mult = None if layer_mult is None else np.ascontiguousarray(layer_mult, np.float32).reshape(L, 2)
        lb = (ctypes.c_float * 8)(*([float(b) for b in level_base] + [0.0] * (8 - len(level_base))))
        self.params = cg_params(len(level_base), lb,
                                None if self._mult is None else self._mult.ctypes.data, R)
        self.n_chunks = -(-S // C) if C > 0 else 0

    @classmethod
    def from_workload(cls, w, **over):
        kw = dict(L=w.L, H=w.H, d=w.d, S=w.S, C=w.C, G=w.G, R=w.R, level_base=w.level_base,
                  layer_mult=w.layer_mult_array())
        kw.update(over)
        return cls(**kw)


# ---- the C ABI, one function each -----------------------------------------
def cg_version() -> int:
    return lib().cg_version()


def cg_status_str(status: int) -> str:
    return lib().cg_status_str(status).decode()


def cg_tables_bytes(cfg: Config) -> int:
    return lib().cg_tables_bytes(ctypes.byref(cfg.dims), ctypes.byref(cfg.params))


def cg_workspace_bytes(cfg: Config, op: int) -> int:
    return lib().cg_workspace_bytes(ctypes.byref(cfg.dims), ctypes.byref(cfg.params), op)


def cg_encode_bound(cfg: Config) -> int:
    v = ctypes.c_uint64(0)
    rc = lib().cg_encode_bound(ctypes.byref(cfg.dims), ctypes.byref(cfg.params), ctypes.byref(v))
    if rc != CG_OK:
        raise CacheGenError(rc, "cg_encode_bound")
    return v.value


def cg_fit_tables(cfg: Config, kv, tables, ws, stream=None) -> int:
    return lib().cg_fit_tables(ctypes.byref(cfg.dims), ctypes.byref(cfg.params), _ptr(kv), _ptr(tables),
                               _ptr(ws), ws.numel() * ws.element_size(), _stream(stream))


def cg_encode(cfg: Config, tables, kv, chunk_levels, out, out_bytes, ws, stream=None) -> int:
    lv = np.ascontiguousarray(np.asarray(chunk_levels, dtype=np.uint8))
    if lv.size != cfg.n_chunks:
        return CG_ERR_INVALID_ARG
    return lib().cg_encode(ctypes.byref(cfg.dims), ctypes.byref(cfg.params), _ptr(tables), _ptr(kv),
                           lv.ctypes.data, _ptr(out), out.numel() * out.element_size(), _ptr(out_bytes),
                           _ptr(ws), ws.numel() * ws.element_size(), _stream(stream))


def cg_assemble(cfg: Config, level_containers, chunk_levels, out, out_bytes, ws, stream=None) -> int:
    """level_containers: one device uint8 tensor per level (None where no
    chunk uses the level), each holding exactly its container's bytes."""
    nl = cfg.params.n_levels
    ptrs = (ctypes.c_void_p * nl)(*[None if c is None else _ptr(c) for c in level_containers])
    sizes = (ctypes.c_uint64 * nl)(*[0 if c is None else c.numel() for c in level_containers])
    lv = np.ascontiguousarray(np.asarray(chunk_levels, dtype=np.uint8))
    if lv.size != cfg.n_chunks or len(level_containers) != nl:
        return CG_ERR_INVALID_ARG
    return lib().cg_assemble(ctypes.byref(cfg.dims), ctypes.byref(cfg.params), ctypes.cast(ptrs, ctypes.c_void_p),
                             ctypes.cast(sizes, ctypes.c_void_p), lv.ctypes.data, _ptr(out),
                             out.numel() * out.element_size(), _ptr(out_bytes), _ptr(ws),
                             ws.numel() * ws.element_size(), _stream(stream))


def cg_decode(cfg: Config, tables, bitstream, nbytes: int, chunk_begin: int, chunk_end: int, kv, ws,
              stream=None) -> int:
    return lib().cg_decode(ctypes.byref(cfg.dims), ctypes.byref(cfg.params), _ptr(tables), _ptr(bitstream),
                           int(nbytes), int(chunk_begin), int(chunk_end), _ptr(kv), _ptr(ws),
                           ws.numel() * ws.element_size(), _stream(stream))


def cg_decode_noalloc(cfg: Config, tables, bitstream, nbytes: int, chunk_begin: int, chunk_end: int, kv,
                      stream=None):
    """cg_decode without a workspace (for callers that cannot allocate).
    Returns (status, device address of the library's scratch, for
    cg_read_status)."""
    addr = ctypes.c_void_p(0)
    rc = lib().cg_decode_noalloc(ctypes.byref(cfg.dims), ctypes.byref(cfg.params), _ptr(tables), _ptr(bitstream),
                                 int(nbytes), int(chunk_begin), int(chunk_end), _ptr(kv), _stream(stream),
                                 ctypes.byref(addr))
    return rc, addr.value


def cg_decode_layers(cfg: Config, tables, bitstream, nbytes: int, chunk_begin: int, chunk_end: int,
                     layer_begin: int, layer_end: int, kv, ws, stream=None) -> int:
    return lib().cg_decode_layers(ctypes.byref(cfg.dims), ctypes.byref(cfg.params), _ptr(tables), _ptr(bitstream),
                                  int(nbytes), int(chunk_begin), int(chunk_end), int(layer_begin), int(layer_end),
                                  _ptr(kv), _ptr(ws), ws.numel() * ws.element_size(), _stream(stream))


def cg_decode_paged(cfg: Config, tables, bitstream, nbytes: int, chunk_begin: int, chunk_end: int, pools,
                    block_table, block_tokens: int, n_blocks: int, ws, stream=None) -> int:
    """cg_decode into a paged cache.  pools: device int64 tensor of the 2*L
    page-pool addresses ([n_blocks][H][block_tokens][d] fp16 each);
    block_table: device int32 tensor of ceil(S / block_tokens) block ids."""
    return lib().cg_decode_paged(ctypes.byref(cfg.dims), ctypes.byref(cfg.params), _ptr(tables), _ptr(bitstream),
                                 int(nbytes), int(chunk_begin), int(chunk_end), _ptr(pools), _ptr(block_table),
                                 int(block_tokens), int(n_blocks), _ptr(ws), ws.numel() * ws.element_size(),
                                 _stream(stream))


class cg_link_step(ctypes.Structure):
    _fields_ = [("seconds", ctypes.c_double), ("bytes_per_s", ctypes.c_double)]


def _link(trace):
    arr = (cg_link_step * len(trace))(*[cg_link_step(float(a), float(b)) for a, b in trace])
    return arr, len(trace)


def cg_plan_levels(chunk_bytes, trace, initial_bytes_per_s: float, deadline_s: float, decode_s):
    """Host-only level controller.  chunk_bytes: [n_chunks][n_levels] ints;
    trace: [(seconds, bytes_per_s)]; decode_s: [n_chunks].
    Returns (status, levels uint8[n], timeline float64[n,3], total seconds)."""
    import numpy as np
    cb = np.ascontiguousarray(chunk_bytes, dtype=np.uint64)
    n, nl = cb.shape
    ds = np.ascontiguousarray(decode_s, dtype=np.float64)
    lv = np.zeros(n, np.uint8)
    tl = np.zeros((n, 3), np.float64)
    tot = ctypes.c_double(0.0)
    arr, ns = _link(trace)
    rc = lib().cg_plan_levels(n, nl, cb.ctypes.data, ctypes.cast(arr, ctypes.c_void_p), ns,
                              float(initial_bytes_per_s), float(deadline_s), ds.ctypes.data, lv.ctypes.data,
                              tl.ctypes.data, ctypes.byref(tot))
    return rc, lv, tl, tot.value


def cg_simulate_stream(chunk_bytes, trace, levels, decode_s):
    """The same link/decode model for given levels -> (status, timeline, total)."""
    import numpy as np
    cb = np.ascontiguousarray(chunk_bytes, dtype=np.uint64)
    n, nl = cb.shape
    ds = np.ascontiguousarray(decode_s, dtype=np.float64)
    lv = np.ascontiguousarray(levels, dtype=np.uint8)
    tl = np.zeros((n, 3), np.float64)
    tot = ctypes.c_double(0.0)
    arr, ns = _link(trace)
    rc = lib().cg_simulate_stream(n, nl, cb.ctypes.data, ctypes.cast(arr, ctypes.c_void_p), ns, lv.ctypes.data,
                                  ds.ctypes.data, tl.ctypes.data, ctypes.byref(tot))
    return rc, tl, tot.value


def cg_entropy_bound(cfg: Config, ws_fit, level: int = 0) -> float:
    """Entropy bound (bytes) of a container with every chunk at `level`,
    from the histograms of the last cg_fit_tables on ws_fit."""
    out = ctypes.c_double(0.0)
    check(lib().cg_entropy_bound(ctypes.byref(cfg.dims), ctypes.byref(cfg.params), _ptr(ws_fit), int(level),
                                 ctypes.byref(out)), "cg_entropy_bound")
    return out.value


def cg_read_status(ws) -> int:
    return lib().cg_read_status(_ptr(ws))


def cg_host_mapped(t) -> int:
    """The device address of a pinned, mapped host tensor (or address), to
    pass as a container or output of the decode calls.  Raises
    CacheGenError when the memory is not pinned and mapped."""
    dp = ctypes.c_void_p(0)
    check(lib().cg_host_mapped(_ptr(t), ctypes.byref(dp)), "cg_host_mapped")
    return int(dp.value)


# ---- buffer helpers (torch allocates; nothing here computes) ----------------
def empty_u8(nbytes: int, device="cuda"):
    """A 256-byte-aligned uint8 device buffer (torch's allocator aligns to 512)."""
    import torch
    return torch.empty(max(int(nbytes), 1), dtype=torch.uint8, device=device)


def check(rc: int, what: str):
    if rc != CG_OK:
        raise CacheGenError(rc, what)
