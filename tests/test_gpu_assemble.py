"""GPU parity of cg_assemble: a mixed-level container built by copying
chunks out of single-level containers (each encoded on the GPU) must equal,
byte for byte, the oracle's encode of the same KV with those levels."""
import numpy as np
import pytest

from kv_cache_compression_02_gb300 import cachegen as cg
from kv_cache_compression_02_gb300 import synth
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu

CASES = {
    "d16_four_levels": (synth.GenSpec(L=4, H=2, d=16, S=700, seed=61, innov="t3", rho=(0.85, 0.99), n_outliers=1,
                                      outlier_scale=20.0), 128, (0.05, 0.1, 0.2, 0.4), [3, 0, 2, 1, 1, 3]),
    "d128_two_of_four_levels": (synth.GenSpec(L=2, H=2, d=128, S=1500, seed=62, innov="t3", rho=(0.85, 0.99)),
                                256, (0.05, 0.1, 0.2, 0.4), [1, 3, 3, 1, 1, 3]),
}


def _setup(orc, name):
    spec, C, lb, lv = CASES[name]
    x = synth.generate(spec)
    cd = orc.Codec(spec.L, spec.H, spec.d, spec.S, C=C, G=10)
    cfg = cg.Config(spec.L, spec.H, spec.d, spec.S, C, G=10, level_base=lb)
    rc, tb = orc.fit_tables(cd, list(lb), None, x)
    assert rc == 0
    levels = np.asarray(lv, np.uint8)
    singles = []
    for level in range(len(lb)):
        if level in lv:
            st, cont, n = gu.encode(cfg, tb, x, np.full(cd.n_chunks, level, np.uint8))
            assert st == cg.CG_OK
            singles.append(gu.to_dev(cont))
        else:
            singles.append(None)
    return cd, cfg, tb, x, levels, singles


def _assemble(cfg, singles, levels, cap):
    T = gu.torch()
    out = cg.empty_u8(cap)
    nb = T.zeros(1, dtype=T.int64, device="cuda")
    ws = cg.empty_u8(cg.cg_workspace_bytes(cfg, cg.CG_OP_ASSEMBLE))
    rc = cg.cg_assemble(cfg, singles, levels, out, nb, ws)
    if rc != cg.CG_OK:
        return rc, None, None
    T.cuda.synchronize()
    n = int(nb.item())
    st = cg.cg_read_status(ws)
    return st, (gu.from_dev(out, n=n) if st == cg.CG_OK else None), n


@pytest.mark.parametrize("name", list(CASES))
def test_assembled_equals_oracle_mixed_encode(orc, name):
    cd, cfg, tb, x, levels, singles = _setup(orc, name)
    rc, want, _ = orc.encode(cd, cfg.params.n_levels, tb, x, levels)
    assert rc == 0
    st, got, n = _assemble(cfg, singles, levels, cg.cg_encode_bound(cfg))
    assert st == cg.CG_OK and n == want.size
    assert np.array_equal(got, want)


def test_assemble_errors(orc):
    cd, cfg, tb, x, levels, singles = _setup(orc, "d16_four_levels")
    # a used level without a container
    assert _assemble(cfg, [singles[0], None, singles[2], singles[3]], levels, 1 << 20)[0] == cg.CG_ERR_INVALID_ARG
    # a container of the wrong level in a slot: its chunk headers disagree
    st, _, _ = _assemble(cfg, [singles[0], singles[2], singles[2], singles[3]], levels, 1 << 20)
    assert st == cg.CG_ERR_CORRUPT
    # too small an output: nothing is copied, the size is reported
    rc, want, _ = orc.encode(cd, 4, tb, x, levels)
    st, _, n = _assemble(cfg, singles, levels, want.size - 16)
    assert st == cg.CG_ERR_CAPACITY and n == want.size
