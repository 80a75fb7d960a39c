"""GPU parity of decoding with host-resident buffers: the container and the
output KV in pinned host memory mapped into the device address space, so
the decoder reads the words and writes the tokens across the host link
(the receiver decodes a streamed context as it arrives: Guide to CacheGen,
pillar 4).  Every result must equal the oracle's decode, bit for bit, with
each d = 128 decoder (a warp per stream with the full tables for 15
chunks and with the u8 tables for 6; the thin-range kernel for a 3-chunk and
a 2-chunk range)."""
import numpy as np
import pytest

from kv_cache_compression_02_gb300 import cachegen as cg
from kv_cache_compression_02_gb300 import synth
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu

FILL = 0x7E00


@pytest.fixture(scope="module")
def case(orc):
    spec = synth.GenSpec(L=2, H=1, d=128, S=14 * 128 + 100, seed=61, innov="t3", rho=(0.85, 0.99),
                         n_outliers=2, outlier_scale=20.0)
    C, G = 128, 10
    x = synth.generate(spec)
    cd = orc.Codec(spec.L, spec.H, spec.d, spec.S, C=C, G=G)
    cfg = cg.Config(spec.L, spec.H, spec.d, spec.S, C, G=G, level_base=(0.1,))
    rc, tb = orc.fit_tables(cd, [0.1], None, x)
    assert rc == 0
    rc, cont, _ = orc.encode(cd, 1, tb, x, np.zeros(cd.n_chunks, np.uint8))
    assert rc == 0
    return spec, cfg, tb, cont


def _host(T, a_u8):
    h = T.empty(a_u8.size, dtype=T.uint8, pin_memory=True)
    h.copy_(T.from_numpy(np.ascontiguousarray(a_u8)))
    return h


def _run(case, k0, k1, layers=None):
    spec, cfg, tb, cont = case
    T = gu.torch()
    gu.ready()
    n = spec.L * 2 * spec.H * spec.S * spec.d
    out = T.full((n,), FILL, dtype=T.int16).pin_memory()
    cont_h = _host(T, cont)
    tbd = gu.to_dev(tb)
    ws = cg.empty_u8(cg.cg_workspace_bytes(cfg, cg.CG_OP_DECODE))
    if layers is None:
        rc = cg.cg_decode(cfg, tbd, gu.host_mapped(cont_h), cont.size, k0, k1, gu.host_mapped(out), ws)
    else:
        rc = cg.cg_decode_layers(cfg, tbd, gu.host_mapped(cont_h), cont.size, k0, k1, layers[0], layers[1],
                                 gu.host_mapped(out), ws)
    assert rc == cg.CG_OK
    T.cuda.synchronize()
    assert cg.cg_read_status(ws) == cg.CG_OK
    return out.numpy().view(np.uint16).reshape(spec.L, 2, spec.H, spec.S, spec.d)


def test_full_decode_host_to_host(orc, case):
    spec, cfg, tb, cont = case
    rc, want = orc.decode(tb, cont)
    assert rc == 0
    assert np.array_equal(_run(case, 0, -1), want)


@pytest.mark.parametrize("k0,k1", [(4, 7), (13, 15), (2, 8)])
def test_chunk_range_host_to_host_writes_only_its_tokens(orc, case, k0, k1):
    spec, cfg, tb, cont = case
    rc, ref = orc.decode(tb, cont, k0, k1)
    assert rc == 0
    t0, t1 = k0 * 128, min(k1 * 128, spec.S)
    want = np.full_like(ref, FILL)
    want[..., t0:t1, :] = ref[..., t0:t1, :]
    assert np.array_equal(_run(case, k0, k1), want)


def test_mapped_address_only_for_page_locked_host_memory(case):
    T = gu.torch()
    gu.ready()
    pinned = T.empty(64, dtype=T.uint8, pin_memory=True)
    assert cg.cg_host_mapped(pinned) != 0
    for t in (T.empty(64, dtype=T.uint8, device="cuda"), T.empty(64, dtype=T.uint8)):  # device, pageable
        with pytest.raises(cg.CacheGenError):
            cg.cg_host_mapped(t)


def test_layer_range_host_to_host(orc, case):
    spec, cfg, tb, cont = case
    rc, ref = orc.decode(tb, cont)
    assert rc == 0
    want = np.full_like(ref, FILL)
    want[1:] = ref[1:]
    assert np.array_equal(_run(case, 0, -1, layers=(1, 2)), want)
