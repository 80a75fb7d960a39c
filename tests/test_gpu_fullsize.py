"""Full-size GPU parity on the four large workloads, every stream.

The GPU fits, encodes and decodes the whole workload in the launch
configuration the benchmark uses.  The oracle then checks, on every host
core (tests/fullverify.py), every chunk stream of every head: the stream
block, scales and int8 anchors byte for byte against its own encode with the
GPU's table rows, the table rows against its own fit, the decoded fp16
tokens against its own decode of the container's streams, and the chunk
index and stream offsets against its stream lengths.  Each container is also held to the entropy bound of its
coded symbols: at most 1% above it (the codec's compression gate).  The
long-context mixed-level workload is also decoded chunk group by chunk group
on a side stream while the next group is copied from pinned host memory, and
must equal the one-shot decode.
"""
import json
import os
import time
from multiprocessing import shared_memory

import numpy as np
import pytest

from kv_cache_compression_02_gb300 import cachegen as cg
from kv_cache_compression_02_gb300 import synth
from kv_cache_compression_02_gb300 import workloads as W
from tests import fullverify
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu


class Run:
    """GPU fit + encode (one container per level set) + decode of a workload;
    the input KV is generated into host shared memory, which the oracle
    workers read."""

    def __init__(self, w):
        T = gu.torch()
        gu.ready()
        self.w = w
        self.shm = shared_memory.SharedMemory(create=True, size=w.fp16_bytes)
        host = np.ndarray(w.elements, np.uint16, buffer=self.shm.buf)
        synth.fill(w.gen, host.ctypes.data)
        self.kv = T.frombuffer(self.shm.buf, dtype=T.int16, count=w.elements).cuda()
        del host
        self.cfg = cg.Config.from_workload(w)
        self.tables = cg.empty_u8(cg.cg_tables_bytes(self.cfg))
        ws = cg.empty_u8(cg.cg_workspace_bytes(self.cfg, cg.CG_OP_FIT))
        cg.check(cg.cg_fit_tables(self.cfg, self.kv, self.tables, ws), "fit")
        T.cuda.synchronize()
        assert cg.cg_read_status(ws) == cg.CG_OK
        del ws

    def close(self):
        self.shm.close()
        self.shm.unlink()

    def encode(self, levels):
        T = gu.torch()
        out = cg.empty_u8(cg.cg_encode_bound(self.cfg))
        nb = T.zeros(1, dtype=T.int64, device="cuda")
        ws = cg.empty_u8(cg.cg_workspace_bytes(self.cfg, cg.CG_OP_ENCODE))
        cg.check(cg.cg_encode(self.cfg, self.tables, self.kv, levels, out, nb, ws), "encode")
        T.cuda.synchronize()
        assert cg.cg_read_status(ws) == cg.CG_OK
        del ws
        n = int(nb.item())
        return out[:n]

    def decode(self, cont_dev, k0=0, k1=-1, out=None):
        T = gu.torch()
        out = T.empty_like(self.kv) if out is None else out
        ws = cg.empty_u8(cg.cg_workspace_bytes(self.cfg, cg.CG_OP_DECODE))
        cg.check(cg.cg_decode(self.cfg, self.tables, cont_dev, cont_dev.numel(), k0, k1, out, ws), "decode")
        T.cuda.synchronize()
        assert cg.cg_read_status(ws) == cg.CG_OK
        return out


def _verify(run, cont, levels, decoded, **kw):
    """Every stream against the oracle; the container within 1% of the
    entropy bound of its coded symbols.  The report is printed (and appended
    as a JSON line to the file CG_FULLVERIFY_OUT names, if set)."""
    t0 = time.time()
    rep = fullverify.verify(run.w, run.tables, cont, levels, decoded, kv_shm=run.shm.name, **kw)
    rep["seconds"] = round(time.time() - t0, 1)
    rep["procs"] = os.cpu_count()
    line = json.dumps({k: v for k, v in rep.items() if k != "errors"} | {"n_errors": len(rep["errors"])})
    print("\n" + line)
    if os.environ.get("CG_FULLVERIFY_OUT"):
        with open(os.environ["CG_FULLVERIFY_OUT"], "a") as fh:
            fh.write(line + "\n")
    assert not rep["errors"], rep["errors"][:20]
    assert rep["actual_over_bound"] <= 1.01, rep
    return rep


@pytest.mark.parametrize("w", [W.LLAMA7B, W.LLAMA3_70B], ids=lambda w: w.name)
def test_fullsize_single_level(w):
    run = Run(w)
    try:
        levels = w.levels_for()
        cont = run.encode(levels)
        decoded = run.decode(cont)
        assert w.fp16_bytes / cont.numel() > 2.5
        _verify(run, cont, levels, decoded)
    finally:
        run.close()


def test_fullsize_three_levels():
    """Llama-3-8B shape: each chunk encoded at all three levels, each
    level's container decoded and checked on its own."""
    w = W.LLAMA3_8B
    run = Run(w)
    try:
        sizes = []
        for lv in range(w.n_levels):
            levels = w.levels_for(lv)
            cont = run.encode(levels)
            decoded = run.decode(cont)
            sizes.append(cont.numel())
            _verify(run, cont, levels, decoded, tables_every=1 if lv == 0 else 1 << 30)
            del decoded, cont
        assert sizes[0] > sizes[1] > sizes[2]  # coarser steps, smaller streams
    finally:
        run.close()


def test_fullsize_mixed_levels_streamed():
    """Long context, one of four levels per chunk; decoded in chunk groups on
    a side stream overlapped with the next group's host-to-device copy."""
    T = gu.torch()
    w = W.LONGCTX_MIXED
    run = Run(w)
    levels = w.levels_for()
    try:
        _streamed(run, levels)
    finally:
        run.close()


def _streamed(run, levels):
    T = gu.torch()
    w = run.w
    cont = run.encode(levels)
    n = cont.numel()
    cont_host = T.empty(n, dtype=T.uint8, pin_memory=True)
    cont_host.copy_(cont)
    one_shot = run.decode(cont)
    ch = cont_host.numpy()
    offs = [int(v) for v in ch[64:64 + 8 * w.n_chunks].view(np.uint64)] + [n]

    dev = cg.empty_u8(n)
    out = T.zeros_like(run.kv)
    ws = cg.empty_u8(cg.cg_workspace_bytes(run.cfg, cg.CG_OP_DECODE))
    copy_s, dec_s = T.cuda.Stream(), T.cuda.Stream()
    streamed = {}
    for group, rep in ((8, 0), (8, 1), (16, 0), (16, 1), (32, 0), (32, 1)):  # the second of each is timed
        out.zero_()
        T.cuda.synchronize()
        t0 = time.perf_counter()
        for g0 in range(0, w.n_chunks, group):
            g1 = min(g0 + group, w.n_chunks)
            lo = 0 if g0 == 0 else offs[g0]
            with T.cuda.stream(copy_s):
                dev[lo:offs[g1]].copy_(cont_host[lo:offs[g1]], non_blocking=True)
                ev = T.cuda.Event()
                ev.record(copy_s)
            dec_s.wait_event(ev)
            cg.check(cg.cg_decode(run.cfg, run.tables, dev, n, g0, g1, out, ws, dec_s), "decode group")
        T.cuda.synchronize()
        if rep:
            streamed[group] = time.perf_counter() - t0
        assert cg.cg_read_status(ws) == cg.CG_OK
        assert T.equal(out, one_shot)
    # the parts alone: the container's host-to-device copy, and the one-shot
    # decode from device memory
    T.cuda.synchronize()
    t0 = time.perf_counter()
    dev.copy_(cont_host, non_blocking=True)
    T.cuda.synchronize()
    t_copy = time.perf_counter() - t0
    t0 = time.perf_counter()
    cg.check(cg.cg_decode(run.cfg, run.tables, dev, n, 0, -1, out, ws), "decode")
    T.cuda.synchronize()
    t_dec = time.perf_counter() - t0
    # one cg_decode reading the container straight from pinned host memory
    out.zero_()
    T.cuda.synchronize()
    t0 = time.perf_counter()
    cg.check(cg.cg_decode(run.cfg, run.tables, cg.cg_host_mapped(cont_host), n, 0, -1, out, ws), "host decode")
    T.cuda.synchronize()
    direct = time.perf_counter() - t0
    assert cg.cg_read_status(ws) == cg.CG_OK
    assert T.equal(out, one_shot)
    print(f"\ncontainer {n / 1e9:.2f} GB; alone: copy {t_copy * 1e3:.1f} ms, decode {t_dec * 1e3:.1f} ms; "
          f"one decode from the pinned host container: {direct * 1e3:.1f} ms "
          f"({w.fp16_bytes / direct / 1e9:.0f} GB/s of fp16)")
    for group, t in streamed.items():
        print(f"streamed decode of {w.n_chunks} chunks in groups of {group}: {t * 1e3:.1f} ms "
              f"({w.fp16_bytes / t / 1e9:.0f} GB/s of fp16); overlap efficiency max(copy, decode) / streamed "
              f"= {max(t_copy, t_dec) / t:.2f}")
    del dev, cont_host
    _verify(run, cont, levels, out)
