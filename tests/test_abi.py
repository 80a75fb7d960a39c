"""The C ABI: the library loads, exports every function include/cachegen.h
declares, and its host-only size queries agree with the oracle (no GPU)."""
import ctypes
import os
import re

import numpy as np
import pytest

from kv_cache_compression_02_gb300 import build, cachegen as cg
from kv_cache_compression_02_gb300 import workloads as W

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    build.build()
    return cg.lib()


def declared_functions():
    names = []
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            src = open(os.path.join(ROOT, "include", fn)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names += re.findall(r"\b(cg_\w+)\s*\(", src)
    return sorted(set(names))


def test_exports_every_declared_symbol(lib):
    names = declared_functions()
    assert len(names) >= 9
    for n in names:
        assert hasattr(lib, n), n


def test_version_and_status_strings(lib):
    assert cg.cg_version() == 1
    assert cg.cg_status_str(cg.CG_ERR_CORRUPT) == "CG_ERR_CORRUPT"
    assert cg.cg_status_str(99) == "CG_ERR_UNKNOWN"


@pytest.mark.parametrize("w", [W.TINY, W.LLAMA7B, W.LLAMA3_8B, W.LLAMA3_70B, W.LONGCTX_MIXED], ids=lambda w: w.name)
def test_sizes_match_oracle(orc, lib, w):
    cfg = cg.Config.from_workload(w)
    cd = orc.Codec(w.L, w.H, w.d, w.S, w.C, w.G, w.R)
    assert cg.cg_tables_bytes(cfg) == orc.tables_bytes(cd, w.n_levels)
    # one word slot per delta symbol per stream, plus the fixed parts
    nk, nstr = w.n_chunks, w.L * 2 * w.H
    pad = lambda v: (v + 15) // 16 * 16  # noqa: E731
    bound = pad(64 + 8 * nk)
    for k in range(nk):
        ntok = min(w.C, w.S - k * w.C)
        ng = -(-ntok // w.G)
        bound += 16 + pad(4 * nstr * w.d) + pad(nstr * ng * w.d) + pad(4 * nstr)
        bound += nstr * pad(16 + 4 * w.d + 2 * (1 if w.R == 127 else 3) * (ntok - ng) * w.d)
    assert cg.cg_encode_bound(cfg) == bound
    for op in (cg.CG_OP_FIT, cg.CG_OP_ENCODE, cg.CG_OP_DECODE):
        assert cg.cg_workspace_bytes(cfg, op) > 0


def test_invalid_arguments(lib):
    bad = [dict(L=1, H=1, d=12, S=10, C=10), dict(L=1, H=1, d=256, S=10, C=10), dict(L=1, H=1, d=8, S=0, C=10),
           dict(L=1, H=1, d=8, S=10, C=0), dict(L=1, H=1, d=8, S=10, C=10, G=0),
           dict(L=1, H=1, d=8, S=10, C=10, R=128), dict(L=1, H=1, d=8, S=2 ** 22 + 1, C=10),
           dict(L=1, H=1, d=8, S=10, C=10, level_base=()), dict(L=1, H=1, d=8, S=10, C=10, level_base=(0.1,) * 9),
           dict(L=1, H=1, d=8, S=10, C=10, level_base=(float("nan"),)),
           dict(L=1, H=1, d=8, S=10, C=10, layer_mult=np.array([[1.0, -1.0]]))]
    for kw in bad:
        lb = kw.pop("level_base", (0.1,))
        if len(lb) > 8:
            continue  # cannot even be expressed in cg_params
        cfg = cg.Config(level_base=lb, **kw)
        if len(lb) == 0:
            cfg.params.n_levels = 0
        assert cg.cg_tables_bytes(cfg) == 0, kw
        assert cg.cg_workspace_bytes(cfg, cg.CG_OP_DECODE) == 0, kw
        with pytest.raises(cg.CacheGenError):
            cg.cg_encode_bound(cfg)
    cfg = cg.Config(L=1, H=1, d=8, S=10, C=10)
    assert cg.cg_workspace_bytes(cfg, 7) == 0
    assert lib.cg_fit_tables(None, None, None, None, None, 0, None) == cg.CG_ERR_INVALID_ARG
    # cg_host_mapped: null pointers are rejected before any CUDA call, and the output is cleared
    dp = ctypes.c_void_p(123)
    assert lib.cg_host_mapped(None, ctypes.byref(dp)) == cg.CG_ERR_INVALID_ARG and not dp.value
    assert lib.cg_host_mapped(ctypes.c_void_p(1 << 20), None) == cg.CG_ERR_INVALID_ARG
    # cg_decode_paged: missing pointers or a block size below 1, rejected before any CUDA call
    ok = cg.Config(L=1, H=1, d=8, S=10, C=10)
    fake = 1 << 20  # an aligned non-null address that is never dereferenced
    args = lambda pools, table, bt, nb: (ctypes.byref(ok.dims), ctypes.byref(ok.params), fake, fake, 4096, 0, -1,  # noqa: E731
                                         pools, table, bt, nb, fake, 1 << 20, None)
    assert lib.cg_decode_paged(*args(None, fake, 4, 4)) == cg.CG_ERR_INVALID_ARG
    assert lib.cg_decode_paged(*args(fake, None, 4, 4)) == cg.CG_ERR_INVALID_ARG
    assert lib.cg_decode_paged(*args(fake, fake, 0, 4)) == cg.CG_ERR_INVALID_ARG
    assert lib.cg_decode_paged(*args(fake, fake, 4, 0)) == cg.CG_ERR_INVALID_ARG
    # cg_assemble: missing arrays or a level out of range, rejected before any CUDA call
    lv = (ctypes.c_uint8 * 1)(0)
    ptrs = (ctypes.c_void_p * 1)(fake)
    sizes = (ctypes.c_uint64 * 1)(1 << 20)
    asm = lambda p, z, l: (ctypes.byref(ok.dims), ctypes.byref(ok.params), p, z, l, fake, 1 << 20, fake,  # noqa: E731
                           fake, 1 << 20, None)
    assert lib.cg_assemble(*asm(None, sizes, lv)) == cg.CG_ERR_INVALID_ARG
    assert lib.cg_assemble(*asm(ptrs, None, lv)) == cg.CG_ERR_INVALID_ARG
    assert lib.cg_assemble(*asm(ptrs, sizes, None)) == cg.CG_ERR_INVALID_ARG
    bad = (ctypes.c_uint8 * 1)(1)  # level 1 of a one-level configuration
    assert lib.cg_assemble(*asm(ptrs, sizes, bad)) == cg.CG_ERR_INVALID_ARG


def test_decode_entry_points_validate_alike(lib):
    """cg_decode and cg_decode_noalloc share their argument checks: a
    non-finite or non-positive layer multiplier (or level base) is rejected by
    both, synchronously and before any CUDA call."""
    fake = 1 << 20  # an aligned non-null address that is never dereferenced
    for mult in (float("nan"), float("inf"), 0.0, -1.0):
        cfg = cg.Config(L=2, H=1, d=8, S=10, C=10, layer_mult=np.array([[1.0, 1.0], [mult, 1.0]], np.float32))
        d, p = ctypes.byref(cfg.dims), ctypes.byref(cfg.params)
        assert lib.cg_decode(d, p, fake, fake, 4096, 0, -1, fake, fake, 1 << 20, None) == cg.CG_ERR_INVALID_ARG
        assert lib.cg_decode_noalloc(d, p, fake, fake, 4096, 0, -1, fake, None, None) == cg.CG_ERR_INVALID_ARG
    cfg = cg.Config(L=1, H=1, d=8, S=10, C=10, level_base=(float("nan"),))
    d, p = ctypes.byref(cfg.dims), ctypes.byref(cfg.params)
    assert lib.cg_decode_noalloc(d, p, fake, fake, 4096, 0, -1, fake, None, None) == cg.CG_ERR_INVALID_ARG
