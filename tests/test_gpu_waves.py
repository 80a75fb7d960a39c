"""GPU parity of the d = 128 full-table decoder when the heads outnumber one
wave of its CTAs (one per SM).  The heads past the last full wave are
decoded by two CTAs each, one on the even and one on the odd entries of the
head's chunk list, when the doubled tail still fits in one wave; the other
heads by one CTA.  A launch that holds both kinds of head, one whose heads
fill whole waves (no pair), and one that is a single short wave (every head
a pair) must each equal the oracle's decode (Guide to CacheGen, pillar 4:
the decoder's output is the encoder's quantised KV, exactly)."""
import numpy as np
import pytest

from kv_cache_compression_02_gb300 import cachegen as cg
from kv_cache_compression_02_gb300 import synth
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu

FILL = 0x7E00


@pytest.fixture(scope="module")
def case(orc):
    T = gu.torch()
    sms = T.cuda.get_device_properties(0).multi_processor_count
    H = 4
    L = sms // (2 * H) + 1  # 2 L H heads = one CTA per SM, plus 1 to 8 heads
    C, G, lb = 128, 10, (0.1,)
    spec = synth.GenSpec(L=L, H=H, d=128, S=10 * C - 37, seed=61, innov="t3", rho=(0.85, 0.99), n_outliers=1,
                         outlier_scale=20.0)
    x = synth.generate(spec)
    cd = orc.Codec(spec.L, spec.H, spec.d, spec.S, C=C, G=G)
    cfg = cg.Config(spec.L, spec.H, spec.d, spec.S, C, G=G, level_base=lb)
    levels = np.zeros(cd.n_chunks, np.uint8)  # one level of ten chunks: the full-table decoder
    rc, tb = orc.fit_tables(cd, list(lb), None, x)
    assert rc == 0
    rc, cont, _ = orc.encode(cd, len(lb), tb, x, levels)
    assert rc == 0
    rc, y_ref = orc.decode(tb, cont)
    assert rc == 0
    return spec, cfg, tb, cont, y_ref, sms


def test_whole_and_paired_heads_in_one_launch(case):
    spec, cfg, tb, cont, y_ref, sms = case
    assert sms < 2 * spec.L * spec.H <= sms + 8
    st, y = gu.decode(cfg, tb, cont, fill=FILL)
    assert st == cg.CG_OK
    assert np.array_equal(y, y_ref)


def _decode_layers(cfg, spec, tb, cont, l0, l1):
    T = gu.torch()
    kv = T.full((spec.L * 2 * spec.H * spec.S * spec.d,), FILL, dtype=T.int16, device="cuda")
    ws = cg.empty_u8(cg.cg_workspace_bytes(cfg, cg.CG_OP_DECODE))
    assert cg.cg_decode_layers(cfg, gu.to_dev(tb), gu.to_dev(cont), cont.size, 0, -1, l0, l1, kv, ws) == cg.CG_OK
    T.cuda.synchronize()
    return cg.cg_read_status(ws), kv.cpu().numpy().view(np.uint16).reshape(spec.L, 2, spec.H, spec.S, spec.d)


@pytest.mark.parametrize("l0, l1", [(0, 1), (1, -1), (2, 5)])
def test_layer_groups_around_the_wave(case, l0, l1):
    """(1, L): the heads of L - 1 layers, one wave or less; (0, 1) and (2, 5):
    a short wave, every head a pair.  Only the group's layers are written."""
    spec, cfg, tb, cont, y_ref, sms = case
    st, y = _decode_layers(cfg, spec, tb, cont, l0, l1)
    assert st == cg.CG_OK
    hi = spec.L if l1 < 0 else l1
    assert np.array_equal(y[l0:hi], y_ref[l0:hi])
    assert (y[:l0] == FILL).all() and (y[hi:] == FILL).all()
