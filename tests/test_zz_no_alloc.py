"""cg_decode_noalloc: the decoder for callers that cannot allocate device
memory (allocator-free runtimes, a device owned by the caller's own pool).

It must decode exactly what cg_decode decodes, twice in a row through the
same shared library scratch, and report its status through that scratch.
This file sorts last so that a run stopping at the first failure has
already run every other test.
"""
import numpy as np
import pytest

from kv_cache_compression_02_gb300 import cachegen as cg
from kv_cache_compression_02_gb300 import synth
from kv_cache_compression_02_gb300 import workloads as W
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu


def test_noalloc_decode_matches_cg_decode():
    gu.ready()
    T = gu.torch()
    w = W.scaled(W.LLAMA3_70B, L=2, H=2, S=5000, C=1536)
    x = synth.generate(w.gen)
    cfg = cg.Config.from_workload(w)
    st, tb = gu.fit(cfg, x)
    assert st == cg.CG_OK
    st, cont, n = gu.encode(cfg, tb, x, w.levels_for())
    assert st == cg.CG_OK
    st, ref = gu.decode(cfg, tb, cont)            # the existing entry point
    assert st == cg.CG_OK

    tbd, buf = gu.to_dev(tb), gu.to_dev(cont)
    for call in range(2):                         # two calls in a row share the scratch
        kv = T.full((x.size,), 0x7E00, dtype=T.int16, device="cuda")
        rc, scratch = cg.cg_decode_noalloc(cfg, tbd, buf, n, 0, -1, kv)
        assert rc == cg.CG_OK and scratch
        T.cuda.synchronize()
        assert cg.cg_read_status(scratch) == cg.CG_OK
        y = kv.cpu().numpy().view(np.uint16).reshape(x.shape)
        assert np.array_equal(y, ref), f"call {call}"

    # a corrupt container is reported through the same scratch, and the next
    # good call clears it
    bad = cont.copy()
    bad[0] ^= 1
    kv = T.zeros(x.size, dtype=T.int16, device="cuda")
    rc, scratch = cg.cg_decode_noalloc(cfg, tbd, gu.to_dev(bad), n, 0, -1, kv)
    T.cuda.synchronize()
    assert rc == cg.CG_OK and cg.cg_read_status(scratch) == cg.CG_ERR_CORRUPT
    rc, scratch = cg.cg_decode_noalloc(cfg, tbd, buf, n, 0, -1, kv)
    T.cuda.synchronize()
    assert rc == cg.CG_OK and cg.cg_read_status(scratch) == cg.CG_OK

    # more chunks than the scratch can list are refused up front
    big = cg.Config(1, 1, 8, 3000, 1, G=1)
    assert cg.cg_decode_noalloc(big, tbd, buf, n, 0, -1, kv)[0] == cg.CG_ERR_CAPACITY
