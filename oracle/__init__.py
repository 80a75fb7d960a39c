"""CPU oracle of the CacheGen KV-cache codec -- TEST INFRASTRUCTURE ONLY.

Only the test suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product path (the CUDA library and
its binding) never loads it, and shares no code with it.

The arithmetic lives in ``cg_oracle.c`` (plain single-threaded C, built with
``-O2 -ffp-contract=off``); this module is ctypes marshalling over numpy
arrays.  Each C function cites the passage of the CacheGen pages it follows.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from dataclasses import dataclass

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "cg_oracle.c")
_LIB = os.path.join(_HERE, "_build", "liborc.so")

OK, ERR_INVALID_ARG, ERR_NONFINITE, ERR_CAPACITY, ERR_CORRUPT = 0, 1, 2, 3, 4
M = 1 << 16
ESC = 255


def build(force: bool = False) -> str:
    """Compile the oracle into ``oracle/_build/liborc.so`` (gcc, no fast-math)."""
    os.makedirs(os.path.dirname(_LIB), exist_ok=True)
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < max(
        os.path.getmtime(_SRC), os.path.getmtime(os.path.join(_HERE, "cg_oracle.h"))
    ):
        tmp = _LIB + f".{os.getpid()}.tmp"
        subprocess.check_call(
            ["gcc", "-O2", "-std=gnu11", "-ffp-contract=off", "-fno-fast-math", "-fPIC",
             "-shared", "-Wall", "-o", tmp, _SRC, "-lm"]
        )
        os.replace(tmp, _LIB)
    return _LIB


class Dims(ctypes.Structure):
    _fields_ = [("L", ctypes.c_int32), ("H", ctypes.c_int32), ("d", ctypes.c_int32),
                ("C", ctypes.c_int32), ("G", ctypes.c_int32), ("R", ctypes.c_int32),
                ("S", ctypes.c_int64)]


class Stats(ctypes.Structure):
    _fields_ = [("entropy_bits", ctypes.c_double), ("n_symbols", ctypes.c_uint64),
                ("n_esc", ctypes.c_uint64), ("n_words", ctypes.c_uint64),
                ("fixed_bytes", ctypes.c_uint64), ("state_bytes", ctypes.c_uint64),
                ("pad_bytes", ctypes.c_uint64)]


_lib = None


def lib():
    global _lib
    if _lib is None:
        _lib = ctypes.CDLL(build())
        P = ctypes.c_void_p
        sig = {
            "orc_f16_to_f32": (ctypes.c_float, [ctypes.c_uint16]),
            "orc_f32_to_f16_rn": (ctypes.c_uint16, [ctypes.c_float]),
            "orc_channel_sigma": (ctypes.c_float, [P, ctypes.c_int64, ctypes.c_int64]),
            "orc_step": (None, [ctypes.c_float, ctypes.c_float, ctypes.c_float, P, P]),
            "orc_anchor_scale": (None, [ctypes.c_float, P, P]),
            "orc_anchor_code": (ctypes.c_int32, [ctypes.c_float, ctypes.c_float, ctypes.c_float, P]),
            "orc_delta_code": (ctypes.c_int32, [ctypes.c_float, ctypes.c_float, ctypes.c_float]),
            "orc_symbol": (ctypes.c_int32, [ctypes.c_int32, ctypes.c_int32]),
            "orc_normalize": (None, [P, P, P]),
            "orc_reconstruct": (ctypes.c_uint16, [ctypes.c_int32, ctypes.c_float, ctypes.c_float]),
            "orc_rans_encode": (ctypes.c_int64, [ctypes.c_int64, ctypes.c_int32, P, P, P, P, P, P]),
            "orc_rans_decode": (ctypes.c_int, [ctypes.c_int64, ctypes.c_int32, P, P, ctypes.c_int64,
                                               ctypes.c_int64, P, P, P, P]),
            "orc_tables_bytes": (ctypes.c_size_t, [P, ctypes.c_int32]),
            "orc_fit_tables": (ctypes.c_int, [P, ctypes.c_int32, P, P, P, P]),
            "orc_fit_head": (ctypes.c_int, [P, ctypes.c_float, ctypes.c_float, P, P, P, P]),
            "orc_encode_stream": (ctypes.c_int64, [P, P, ctypes.c_int64, P, P, P, P, P, P,
                                                   ctypes.c_int64, P, P]),
            "orc_encode_bound": (ctypes.c_uint64, [P]),
            "orc_table_entropy": (ctypes.c_double, [P]),
            "orc_container_fixed_bytes": (ctypes.c_uint64, [P]),
            "orc_encode": (ctypes.c_int, [P, ctypes.c_int32, P, P, P, P, ctypes.c_uint64, P, P]),
            "orc_decode": (ctypes.c_int, [P, ctypes.c_size_t, P, ctypes.c_uint64, ctypes.c_int64,
                                          ctypes.c_int64, P]),
            "orc_decode_stream": (ctypes.c_int, [P, P, ctypes.c_uint64, ctypes.c_int64, P, P, P, P, P]),
        }
        for name, (res, args) in sig.items():
            fn = getattr(_lib, name)
            fn.restype = res
            fn.argtypes = args
    return _lib


def _p(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data_as(ctypes.c_void_p)


def _ref(x):
    return ctypes.cast(ctypes.pointer(x), ctypes.c_void_p)


@dataclass(frozen=True)
class Codec:
    """Geometry and codec parameters (the oracle's own copy)."""
    L: int
    H: int
    d: int
    S: int
    C: int
    G: int = 10
    R: int = 127

    def dims(self) -> Dims:
        return Dims(self.L, self.H, self.d, self.C, self.G, self.R, self.S)

    @property
    def n_chunks(self) -> int:
        return -(-self.S // self.C)


# ---- scalar steps ---------------------------------------------------------
def f16_to_f32(h: int) -> float:
    return lib().orc_f16_to_f32(h)


def f32_to_f16(f: float) -> int:
    return lib().orc_f32_to_f16_rn(np.float32(f))


def channel_sigma(x_f16: np.ndarray) -> np.float32:
    x = np.ascontiguousarray(x_f16, dtype=np.uint16)
    return np.float32(lib().orc_channel_sigma(_p(x), x.size, 1))


def step(base, mult, sigma):
    s, r = ctypes.c_float(), ctypes.c_float()
    lib().orc_step(np.float32(base), np.float32(mult), np.float32(sigma), _ref(s), _ref(r))
    return np.float32(s.value), np.float32(r.value)


def anchor_scale(absmax):
    s, i = ctypes.c_float(), ctypes.c_float()
    lib().orc_anchor_scale(np.float32(absmax), _ref(s), _ref(i))
    return np.float32(s.value), np.float32(i.value)


def anchor_code(x, s, inv):
    a = ctypes.c_float()
    q = lib().orc_anchor_code(np.float32(x), np.float32(s), np.float32(inv), _ref(a))
    return q, np.float32(a.value)


def delta_code(x, ahat, recip) -> int:
    return lib().orc_delta_code(np.float32(x), np.float32(ahat), np.float32(recip))


def symbol(q, R=127) -> int:
    return lib().orc_symbol(int(q), int(R))


def reconstruct(q, step_, ahat) -> int:
    return lib().orc_reconstruct(int(q), np.float32(step_), np.float32(ahat))


def normalize(counts: np.ndarray):
    n = np.ascontiguousarray(counts, dtype=np.uint64)
    assert n.shape == (256,)
    f = np.zeros(256, np.uint32)
    c = np.zeros(257, np.uint32)
    lib().orc_normalize(_p(n), _p(f), _p(c))
    return f, c


def rans_encode(sym: np.ndarray, q: np.ndarray, f: np.ndarray, cdf: np.ndarray):
    """sym,q: [n][d]; f: [d][256]; cdf: [d][257] -> (states[d], words)."""
    sym = np.ascontiguousarray(sym, np.uint8)
    q = np.ascontiguousarray(q, np.int32)
    n, d = sym.shape
    f = np.ascontiguousarray(f, np.uint32)
    cdf = np.ascontiguousarray(cdf, np.uint32)
    st = np.zeros(d, np.uint32)
    w = np.zeros(3 * n * d + 1, np.uint16)
    nw = lib().orc_rans_encode(n, d, _p(sym), _p(q), _p(f), _p(cdf), _p(st), _p(w))
    return st, w[:nw].copy()


def rans_decode(n: int, states, words, n_esc, f, cdf):
    st = np.ascontiguousarray(states, np.uint32)
    d = st.size
    w = np.ascontiguousarray(words, np.uint16)
    if w.size == 0:
        w = np.zeros(1, np.uint16)
        nw = 0
    else:
        nw = w.size
    f = np.ascontiguousarray(f, np.uint32)
    cdf = np.ascontiguousarray(cdf, np.uint32)
    sym = np.zeros((max(n, 1), d), np.uint8)
    q = np.zeros((max(n, 1), d), np.int32)
    rc = lib().orc_rans_decode(n, d, _p(st), _p(w), nw, int(n_esc), _p(f), _p(cdf), _p(sym), _p(q))
    return rc, sym[:n], q[:n]


# ---- container level ------------------------------------------------------
def tables_bytes(cd: Codec, n_levels: int) -> int:
    return lib().orc_tables_bytes(_ref(cd.dims()), n_levels)


def fit_tables(cd: Codec, level_base, layer_mult, kv: np.ndarray):
    """kv: uint16 [L,2,H,S,d].  Returns (rc, tables uint8)."""
    kv = np.ascontiguousarray(kv, np.uint16)
    nl = len(level_base)
    lb = np.zeros(8, np.float32)
    lb[:nl] = level_base
    lm = None if layer_mult is None else np.ascontiguousarray(layer_mult, np.float32)
    tb = np.zeros(tables_bytes(cd, nl), np.uint8)
    rc = lib().orc_fit_tables(_ref(cd.dims()), nl, _p(lb), None if lm is None else _p(lm), _p(kv), _p(tb))
    return rc, tb


def fit_head(cd: Codec, base, mult, head: np.ndarray):
    """head: uint16 [S][d] -> (rc, step[d], recip[d], cdf[d][256])."""
    head = np.ascontiguousarray(head, np.uint16)
    st = np.zeros(cd.d, np.float32)
    rp = np.zeros(cd.d, np.float32)
    cdf = np.zeros((cd.d, 256), np.uint16)
    rc = lib().orc_fit_head(_ref(cd.dims()), np.float32(base), np.float32(mult), _p(head),
                            _p(st), _p(rp), _p(cdf))
    return rc, st, rp, cdf


def encode_stream(cd: Codec, head, k, step_, recip, cdf, symcount=None, stats=None):
    """Encode chunk k of one head -> (rc_or_len, block bytes, s[d], anchors[ng][d]).
    symcount (uint64 [d][256]) accumulates the coded symbols per lane's
    table; stats (Stats) accumulates the stream's size split."""
    head = np.ascontiguousarray(head, np.uint16)
    ntok = min(cd.C, cd.S - k * cd.C)
    ng = -(-ntok // cd.G)
    cap = 16 + 4 * cd.d + 6 * ntok * cd.d + 32
    blk = np.zeros(cap, np.uint8)
    s = np.zeros(cd.d, np.float32)
    anc = np.zeros((ng, cd.d), np.int8)
    n = lib().orc_encode_stream(_ref(cd.dims()), _p(head), k, _p(np.ascontiguousarray(step_, np.float32)),
                                _p(np.ascontiguousarray(recip, np.float32)),
                                _p(np.ascontiguousarray(cdf, np.uint16)), _p(s), _p(anc), _p(blk), cap,
                                None if symcount is None else _p(symcount), None if stats is None else _ref(stats))
    return n, (blk[:n].copy() if n > 0 else None), s, anc


def encode_bound(cd: Codec) -> int:
    return lib().orc_encode_bound(_ref(cd.dims()))


def encode(cd: Codec, n_levels: int, tables: np.ndarray, kv: np.ndarray, chunk_level):
    """Returns (rc, container uint8, Stats)."""
    kv = np.ascontiguousarray(kv, np.uint16)
    lv = np.ascontiguousarray(np.asarray(chunk_level, dtype=np.uint8))
    assert lv.size == cd.n_chunks
    cap = encode_bound(cd)
    out = np.zeros(cap, np.uint8)
    nbytes = ctypes.c_uint64(0)
    st = Stats()
    rc = lib().orc_encode(_ref(cd.dims()), n_levels, _p(np.ascontiguousarray(tables, np.uint8)), _p(kv),
                          _p(lv), _p(out), cap, _ref(nbytes), _ref(st))
    return rc, out[: nbytes.value].copy(), st


def decode(tables: np.ndarray, container: np.ndarray, k0: int = 0, k1: int | None = None, out=None):
    """Decode chunks [k0,k1) into out ([L,2,H,S,d] uint16, zeros if None)."""
    buf = np.ascontiguousarray(container, np.uint8)
    L, H, d = (int(v) for v in buf[8:20].view(np.uint32))
    S = int(buf[32:40].view(np.uint64)[0])
    nk = int(buf[44:48].view(np.uint32)[0])
    if k1 is None:
        k1 = nk
    if out is None:
        out = np.zeros((L, 2, H, S, d), np.uint16)
    tb = np.ascontiguousarray(tables, np.uint8)
    rc = lib().orc_decode(_p(tb), tb.size, _p(buf), buf.size, k0, k1, _p(out))
    return rc, out


def paged_from_contiguous(kv: np.ndarray, block_table, block_tokens: int, n_blocks: int, fill: int = 0,
                          tokens=None) -> np.ndarray:
    """The paged cache that holds kv ([L,2,H,S,d] uint16): pools
    [L][2][n_blocks][H][block_tokens][d], token t of the sequence at row
    t % block_tokens of block block_table[t // block_tokens] (the block-table
    layout the Guide to CacheGen's deployment notes name for paged-attention
    servers).  Rows no token maps to keep `fill`.  tokens: the token indices
    to place (default all S)."""
    L, _, H, S, d = kv.shape
    pools = np.full((L, 2, n_blocks, H, block_tokens, d), fill, np.uint16)
    for t in (range(S) if tokens is None else tokens):
        b = int(block_table[t // block_tokens])
        pools[:, :, b, :, t % block_tokens, :] = kv[:, :, :, t, :]
    return pools


def decode_stream(cd: Codec, blk, k, step_, cdf, s, anchors, head_out):
    blk = np.ascontiguousarray(blk, np.uint8)
    return lib().orc_decode_stream(_ref(cd.dims()), _p(blk), blk.size, k,
                                   _p(np.ascontiguousarray(step_, np.float32)),
                                   _p(np.ascontiguousarray(cdf, np.uint16)),
                                   _p(np.ascontiguousarray(s, np.float32)),
                                   _p(np.ascontiguousarray(anchors, np.int8)), _p(head_out))


def tables_views(tables: np.ndarray, cd: Codec, n_levels: int):
    """(step, recip, cdf) views of a tables blob: [NL][L][2][H*d](...)."""
    nc = n_levels * cd.L * 2 * cd.H * cd.d
    pad = lambda v: (v + 15) & ~15  # noqa: E731
    o1 = 64
    o2 = o1 + pad(4 * nc)
    o3 = o2 + pad(4 * nc)
    shp = (n_levels, cd.L, 2, cd.H * cd.d)
    step_ = tables[o1:o1 + 4 * nc].view(np.float32).reshape(shp)
    recip = tables[o2:o2 + 4 * nc].view(np.float32).reshape(shp)
    cdf = tables[o3:o3 + 512 * nc].view(np.uint16).reshape(shp + (256,))
    return step_, recip, cdf


def table_entropy(counts: np.ndarray) -> float:
    """sum_s n_s log2(N / n_s) (bits) of one table's 256 symbol counts."""
    c = np.ascontiguousarray(counts, np.uint64)
    assert c.shape == (256,)
    return lib().orc_table_entropy(_p(c))


def container_fixed_bytes(cd: Codec) -> int:
    """Header, index and per-chunk fixed parts of a container, unpadded (the
    structural term of the entropy bound; stream headers are counted per
    stream by encode_stream's stats)."""
    return lib().orc_container_fixed_bytes(_ref(cd.dims()))


def entropy_bound_bytes(st: Stats, table_bytes: int = 0) -> float:
    """Entropy of the coded symbols (bits/8) + raw escapes + information-
    bearing structural bytes (+ tables when given)."""
    return st.entropy_bits / 8.0 + 4.0 * st.n_esc + st.fixed_bytes + table_bytes
