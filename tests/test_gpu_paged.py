"""GPU parity of cg_decode_paged: decoding straight into a block-table
paged cache (the Guide to CacheGen's deployment notes: integrating with
PagedAttention, direct paged buffer injection).  The expected cache is the
oracle's decode placed by the block-table definition; every byte,
including rows no token maps to, is compared."""
import numpy as np
import pytest

from kv_cache_compression_02_gb300 import cachegen as cg
from kv_cache_compression_02_gb300 import synth
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu

FILL = 0x7E00  # an fp16 NaN: rows the decode must not touch keep it

CASES = {
    # name: (GenSpec, C, G, level_base, chunk levels, block_tokens, extra blocks, chunk range)
    "d128_bt16_shuffled": (synth.GenSpec(L=2, H=2, d=128, S=3000, seed=41, innov="t3", rho=(0.85, 0.99),
                                         outlier_frac=0.01, outlier_scale=20.0), 1024, 10, (0.1,), None, 16, 7,
                           (0, -1)),
    "d8_bt7_chunk_range": (synth.GenSpec(L=3, H=3, d=8, S=333, seed=42, innov="laplace", rho=(0.95, 0.95),
                                         n_outliers=1), 50, 7, (0.2,), None, 7, 3, (1, 4)),
    "d16_bt1_mixed_levels": (synth.GenSpec(L=2, H=2, d=16, S=300, seed=43, innov="t3", rho=(0.85, 0.99),
                                           n_outliers=1), 64, 10, (0.05, 0.4), [1, 0, 1, 1, 0], 1, 0, (0, -1)),
    "d64_one_block_longer_than_S": (synth.GenSpec(L=1, H=2, d=64, S=250, seed=44), 100, 10, (0.1,), None, 512, 2,
                                    (0, -1)),
    # d = 128, six chunks of one level: a warp per stream with the u8 tables
    "d128_bt16_mid_range": (synth.GenSpec(L=2, H=2, d=128, S=1500, seed=46, innov="t3", rho=(0.85, 0.99),
                                          n_outliers=1, outlier_scale=20.0), 256, 10, (0.1,), None, 16, 4,
                            (0, -1)),
    # d = 128, four chunks of two levels: the thin-range decoder
    "d128_bt16_thin_range": (synth.GenSpec(L=2, H=2, d=128, S=1500, seed=45, innov="t3", rho=(0.85, 0.99),
                                           n_outliers=1, outlier_scale=20.0), 256, 10, (0.1, 0.3),
                             [0, 1, 0, 1, 1, 0], 16, 5, (1, 5)),
}


def _run(orc, name, corrupt_block=None):
    T = gu.torch()
    spec, C, G, lb, lv, bt, extra, (k0, k1) = CASES[name]
    x = synth.generate(spec)
    cd = orc.Codec(spec.L, spec.H, spec.d, spec.S, C=C, G=G)
    cfg = cg.Config(spec.L, spec.H, spec.d, spec.S, C, G=G, level_base=lb)
    levels = np.zeros(cd.n_chunks, np.uint8) if lv is None else np.asarray(lv, np.uint8)
    rc, tb = orc.fit_tables(cd, list(lb), None, x)
    assert rc == 0
    rc, cont, _ = orc.encode(cd, len(lb), tb, x, levels)
    assert rc == 0
    kend = cd.n_chunks if k1 < 0 else k1
    rc, y_ref = orc.decode(tb, cont, k0, kend)
    assert rc == 0
    n_lblk = -(-spec.S // bt)
    n_blocks = n_lblk + extra
    rng = np.random.default_rng(7)
    table = rng.permutation(n_blocks)[:n_lblk].astype(np.int32)
    if corrupt_block is not None:
        table[corrupt_block] = n_blocks  # out of range
    tokens = range(k0 * C, min(kend * C, spec.S))
    L, H, d = spec.L, spec.H, spec.d
    pools = T.full((L * 2, n_blocks, H, bt, d), FILL, dtype=T.int16, device="cuda")
    stride = n_blocks * H * bt * d * 2
    ptrs = T.tensor([pools.data_ptr() + i * stride for i in range(L * 2)], dtype=T.int64, device="cuda")
    tab = T.from_numpy(table).cuda()
    ws = cg.empty_u8(cg.cg_workspace_bytes(cfg, cg.CG_OP_DECODE))
    tb_dev, cont_dev = gu.to_dev(tb), gu.to_dev(cont)
    rc = cg.cg_decode_paged(cfg, tb_dev, cont_dev, cont.size, k0, k1, ptrs, tab, bt, n_blocks, ws)
    assert rc == cg.CG_OK
    T.cuda.synchronize()
    st = cg.cg_read_status(ws)
    got = pools.cpu().numpy().view(np.uint16).reshape(L, 2, n_blocks, H, bt, d)
    return st, got, y_ref, table, tokens, bt, n_blocks


@pytest.mark.parametrize("name", list(CASES))
def test_paged_decode_bit_exact(orc, name):
    st, got, y_ref, table, tokens, bt, n_blocks = _run(orc, name)
    assert st == cg.CG_OK
    want = orc.paged_from_contiguous(y_ref, table, bt, n_blocks, fill=FILL, tokens=tokens)
    if not np.array_equal(got, want):
        bad = np.argwhere(got != want)
        pytest.fail(f"{len(bad)} fp16 values differ, first at {bad[:4].tolist()}")


def test_paged_decode_bad_block_id(orc):
    """An out-of-range block id is reported as an invalid argument; its rows
    are not written, every other row is still exact."""
    st, got, y_ref, table, tokens, bt, n_blocks = _run(orc, "d128_bt16_shuffled", corrupt_block=5)
    assert st == cg.CG_ERR_INVALID_ARG
    ok_tokens = [t for t in tokens if t // bt != 5]
    want = orc.paged_from_contiguous(y_ref, np.where(table < n_blocks, table, 0), bt, n_blocks, fill=FILL,
                                     tokens=ok_tokens)
    assert np.array_equal(got, want)


def test_paged_rejects_bad_arguments(orc):
    spec = CASES["d8_bt7_chunk_range"][0]
    cfg = cg.Config(spec.L, spec.H, spec.d, spec.S, 50, G=7, level_base=(0.2,))
    T = gu.torch()
    buf = cg.empty_u8(4096)
    ws = cg.empty_u8(cg.cg_workspace_bytes(cfg, cg.CG_OP_DECODE))
    ptrs = T.zeros(spec.L * 2, dtype=T.int64, device="cuda")
    tab = T.zeros(64, dtype=T.int32, device="cuda")
    for bt, nb in ((0, 4), (7, 0), (-3, 4)):
        assert cg.cg_decode_paged(cfg, buf, buf, 4096, 0, -1, ptrs, tab, bt, nb, ws) == cg.CG_ERR_INVALID_ARG
    assert cg.cg_decode_paged(cfg, buf, buf, 4096, 0, -1, None, tab, 7, 4, ws) == cg.CG_ERR_INVALID_ARG
