"""GPU parity of cg_decode_layers: decoding a container layer group by
layer group, in execution order (Guide to CacheGen, pillar 4: layer 0
first, so generation can start before the last layer is decoded).  Every
group's output must equal the oracle's decode of those layers, and nothing
outside the group may be written."""
import numpy as np
import pytest

from kv_cache_compression_02_gb300 import cachegen as cg
from kv_cache_compression_02_gb300 import synth
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu

FILL = 0x7E00


@pytest.fixture(scope="module")
def case(orc):
    spec = synth.GenSpec(L=5, H=2, d=16, S=700, seed=51, innov="t3", rho=(0.85, 0.99), n_outliers=1,
                         outlier_scale=20.0)
    C, G, lb = 128, 10, (0.05, 0.2)
    x = synth.generate(spec)
    cd = orc.Codec(spec.L, spec.H, spec.d, spec.S, C=C, G=G)
    cfg = cg.Config(spec.L, spec.H, spec.d, spec.S, C, G=G, level_base=lb)
    levels = np.array([1, 0, 0, 1, 1, 0], np.uint8)
    rc, tb = orc.fit_tables(cd, list(lb), None, x)
    assert rc == 0
    rc, cont, _ = orc.encode(cd, len(lb), tb, x, levels)
    assert rc == 0
    return spec, cfg, cd, tb, cont


def _decode_groups(cfg, spec, tb, cont, groups, k0=0, k1=-1):
    T = gu.torch()
    kv = T.full((spec.L * 2 * spec.H * spec.S * spec.d,), FILL, dtype=T.int16, device="cuda")
    tbd, cd_ = gu.to_dev(tb), gu.to_dev(cont)
    ws = cg.empty_u8(cg.cg_workspace_bytes(cfg, cg.CG_OP_DECODE))
    sts = []
    for l0, l1 in groups:
        assert cg.cg_decode_layers(cfg, tbd, cd_, cont.size, k0, k1, l0, l1, kv, ws) == cg.CG_OK
        T.cuda.synchronize()
        sts.append(cg.cg_read_status(ws))
    return sts, kv.cpu().numpy().view(np.uint16).reshape(spec.L, 2, spec.H, spec.S, spec.d)


def test_layer_groups_cover_the_full_decode(orc, case):
    spec, cfg, cd, tb, cont = case
    rc, y_ref = orc.decode(tb, cont)
    assert rc == 0
    sts, y = _decode_groups(cfg, spec, tb, cont, [(0, 2), (2, 3), (3, -1)])
    assert sts == [cg.CG_OK] * 3
    assert np.array_equal(y, y_ref)


def test_layer_group_and_chunk_range_write_only_their_tokens(orc, case):
    spec, cfg, cd, tb, cont = case
    rc, y_ref = orc.decode(tb, cont, 2, 4)
    assert rc == 0
    sts, y = _decode_groups(cfg, spec, tb, cont, [(1, 3)], k0=2, k1=4)
    assert sts == [cg.CG_OK]
    want = np.full_like(y_ref, FILL)
    want[1:3, :, :, 2 * 128:4 * 128] = y_ref[1:3, :, :, 2 * 128:4 * 128]
    assert np.array_equal(y, want)


def test_empty_and_invalid_layer_ranges(case):
    spec, cfg, cd, tb, cont = case
    T = gu.torch()
    kv = T.full((spec.L * 2 * spec.H * spec.S * spec.d,), FILL, dtype=T.int16, device="cuda")
    tbd, cd_ = gu.to_dev(tb), gu.to_dev(cont)
    ws = cg.empty_u8(cg.cg_workspace_bytes(cfg, cg.CG_OP_DECODE))
    for l0, l1 in ((3, 2), (-1, 2), (0, spec.L + 1), (spec.L + 1, -1)):
        assert cg.cg_decode_layers(cfg, tbd, cd_, cont.size, 0, -1, l0, l1, kv, ws) == cg.CG_ERR_INVALID_ARG
    assert cg.cg_decode_layers(cfg, tbd, cd_, cont.size, 0, -1, 2, 2, kv, ws) == cg.CG_OK  # nothing to do
    T.cuda.synchronize()
    assert (kv.cpu().numpy().view(np.uint16) == FILL).all()


def test_layer_groups_d128_thin_range(orc):
    """Layer groups of a short chunk range at d = 128 (the thin-range
    decoder): each group's tokens equal the oracle's, the rest is untouched."""
    spec = synth.GenSpec(L=3, H=1, d=128, S=600, seed=52, innov="t3", rho=(0.85, 0.99), n_outliers=1,
                         outlier_scale=20.0)
    C, G, lb = 128, 10, (0.05, 0.2)
    x = synth.generate(spec)
    cd = orc.Codec(spec.L, spec.H, spec.d, spec.S, C=C, G=G)
    cfg = cg.Config(spec.L, spec.H, spec.d, spec.S, C, G=G, level_base=lb)
    levels = np.array([1, 0, 0, 1, 1], np.uint8)
    rc, tb = orc.fit_tables(cd, list(lb), None, x)
    assert rc == 0
    rc, cont, _ = orc.encode(cd, len(lb), tb, x, levels)
    assert rc == 0
    rc, y_ref = orc.decode(tb, cont, 1, 4)
    assert rc == 0
    sts, y = _decode_groups(cfg, spec, tb, cont, [(1, 2), (2, 3)], k0=1, k1=4)
    assert sts == [cg.CG_OK] * 2
    t0, t1 = 1 * C, 4 * C
    assert np.array_equal(y[1:, :, :, t0:t1], y_ref[1:, :, :, t0:t1])
    assert (y[0] == FILL).all()
    assert (y[:, :, :, :t0] == FILL).all() and (y[:, :, :, t1:] == FILL).all()
