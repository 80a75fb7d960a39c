"""The full-size parity pass (tests/fullverify.py) on the CPU: handed the
oracle's own tables, container and decode of a small workload as if they
came from the GPU, it finds no difference and its entropy bound equals the
oracle's whole-container figure; a planted change to one stream byte, to a
decoded value or to a stream offset is reported."""
import numpy as np
import pytest
import torch

from kv_cache_compression_02_gb300 import synth
from kv_cache_compression_02_gb300 import workloads as W
from tests import fullverify


@pytest.fixture(scope="module")
def small(orc):
    w = W.scaled(W.LONGCTX_MIXED, L=2, H=2, S=5000, C=1024, name="fullverify_small")
    x = synth.generate(w.gen)
    cd = orc.Codec(w.L, w.H, w.d, w.S, w.C, w.G, w.R)
    rc, tb = orc.fit_tables(cd, list(w.level_base), None, x)
    assert rc == 0
    levels = w.levels_for()
    assert len(set(levels.tolist())) > 1
    rc, cont, st = orc.encode(cd, w.n_levels, tb, x, levels)
    assert rc == 0
    rc, y = orc.decode(tb, cont)
    assert rc == 0
    return w, torch.from_numpy(tb), torch.from_numpy(cont), levels, torch.from_numpy(y.view(np.int16).reshape(-1)), st


def test_clean_container_and_bound(orc, small):
    w, tb, cont, levels, dec, st = small
    rep = fullverify.verify(w, tb, cont, levels, dec, procs=2, batch=3)
    assert rep["errors"] == []
    assert rep["escapes"] == st.n_esc
    assert abs(rep["bound_bytes"] - orc.entropy_bound_bytes(st)) <= 1e-9 * rep["bound_bytes"]
    assert 1.0 <= rep["actual_over_bound"] < 1.05  # short streams: the 4-byte flush per lane weighs more


def test_planted_differences_are_reported(small):
    w, tb, cont, levels, dec, st = small
    bad = cont.clone()
    base = int(bad[64:72].numpy().view(np.uint64)[0])
    nstr = w.L * 2 * w.H
    ng = -(-min(w.C, w.S) // w.G)
    sec_off = 16 + (4 * nstr * w.d + 15) // 16 * 16 + (nstr * ng * w.d + 15) // 16 * 16
    so = int(bad[base + sec_off + 4:base + sec_off + 8].numpy().view(np.uint32)[0])  # stream 1 of chunk 0
    bad[base + so + 16 + 4 * w.d + 3] ^= 1  # a word of that stream
    rep = fullverify.verify(w, tb, bad, levels, dec, procs=2, batch=3)
    assert any("stream of head 1 chunk 0" in e for e in rep["errors"])
    dbad = dec.clone()
    dbad[w.S * w.d * 2 + 5] += 1  # head 2, token 0, lane 5
    rep = fullverify.verify(w, tb, cont, levels, dbad, procs=2, batch=3)
    assert rep["errors"] and all("decoded head 2" in e for e in rep["errors"])
    obad = cont.clone()
    obad[base + sec_off + 8] += 16  # stream 2's offset in chunk 0
    rep = fullverify.verify(w, tb, obad, levels, dec, procs=2, batch=3)
    assert any("chunk 0 stream offsets" in e for e in rep["errors"])
