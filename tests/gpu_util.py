"""Helpers for the GPU tests: run the C-ABI calls on numpy inputs and bring
the results back.  Device memory comes from torch; every computation runs
in libcachegen.so."""
from __future__ import annotations

import numpy as np

from kv_cache_compression_02_gb300 import build, cachegen as cg


def torch():
    import torch as _t
    return _t


def ready():
    build.build()
    cg.lib()


def to_dev(a: np.ndarray):
    t = torch()
    return t.from_numpy(np.ascontiguousarray(a).view(np.uint8).reshape(-1)).cuda()


def from_dev(t, dtype=np.uint8, n=None) -> np.ndarray:
    a = t.cpu().numpy()
    if n is not None:
        a = a[:n]
    return a.view(dtype)


def fit(cfg: cg.Config, kv: np.ndarray):
    """-> (status, tables uint8)"""
    T = torch()
    kvd = to_dev(kv)
    tb = cg.empty_u8(cg.cg_tables_bytes(cfg))
    ws = cg.empty_u8(cg.cg_workspace_bytes(cfg, cg.CG_OP_FIT))
    cg.check(cg.cg_fit_tables(cfg, kvd, tb, ws), "cg_fit_tables")
    T.cuda.synchronize()
    return cg.cg_read_status(ws), from_dev(tb)


def encode(cfg: cg.Config, tables: np.ndarray, kv: np.ndarray, levels, cap: int | None = None):
    """-> (status, container uint8 (None if it did not fit), reported size)"""
    T = torch()
    kvd = to_dev(kv)
    tb = to_dev(tables)
    cap = cg.cg_encode_bound(cfg) if cap is None else cap
    out = cg.empty_u8(cap)
    nb = T.zeros(1, dtype=T.int64, device="cuda")
    ws = cg.empty_u8(cg.cg_workspace_bytes(cfg, cg.CG_OP_ENCODE))
    cg.check(cg.cg_encode(cfg, tb, kvd, levels, out, nb, ws), "cg_encode")
    T.cuda.synchronize()
    st = cg.cg_read_status(ws)
    n = int(nb.item())
    return st, (from_dev(out, n=n) if st == cg.CG_OK else None), n


def decode(cfg: cg.Config, tables: np.ndarray, cont: np.ndarray, k0=0, k1=-1, nbytes=None, fill=0):
    """-> (status, kv uint16 [L,2,H,S,d])"""
    T = torch()
    L, H, d, S = cfg.dims.L, cfg.dims.H, cfg.dims.d, cfg.dims.S
    tb = to_dev(tables)
    buf = to_dev(cont)
    kv = T.full((L * 2 * H * S * d,), fill, dtype=T.int16, device="cuda")
    ws = cg.empty_u8(cg.cg_workspace_bytes(cfg, cg.CG_OP_DECODE))
    rc = cg.cg_decode(cfg, tb, buf, cont.size if nbytes is None else nbytes, k0, k1, kv, ws)
    if rc != cg.CG_OK:
        return rc, None
    T.cuda.synchronize()
    return cg.cg_read_status(ws), kv.cpu().numpy().view(np.uint16).reshape(L, 2, H, S, d)


def host_mapped(t) -> int:
    """The device address of a pinned host tensor (the library's cg_host_mapped)."""
    return cg.cg_host_mapped(t)
