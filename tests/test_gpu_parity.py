"""GPU parity: libcachegen.so against the CPU oracle, element by element.

Tables, containers and decoded fp16 must be bit-identical (the method fixes
every rounding: fp32 multiply by a stored reciprocal, one fma, RN
conversions; sigma from exact integer moments).  Sizes span several tiles,
chunks and anchor groups with ragged tails, every supported head dim, the
escape path, mixed per-chunk levels and the degenerate shapes.
"""
import numpy as np
import pytest

from kv_cache_compression_02_gb300 import cachegen as cg
from kv_cache_compression_02_gb300 import synth
from kv_cache_compression_02_gb300 import workloads as W
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    gu.ready()


CASES = {
    # name: (GenSpec, C, G, R, level_base, layer_mult, chunk levels)
    "tiny_workload": (W.TINY.gen, W.TINY.C, 10, 127, (0.1,), W.TINY.layer_mult_array(), None),
    "d128_ragged_chunks": (synth.GenSpec(L=2, H=2, d=128, S=3000, seed=21, innov="t3", rho=(0.85, 0.99),
                                         outlier_frac=0.01, outlier_scale=20.0), 1024, 10, 127, (0.1,), None, None),
    "d8_group7": (synth.GenSpec(L=3, H=3, d=8, S=333, seed=22, innov="laplace", rho=(0.95, 0.95), n_outliers=1),
                  50, 7, 127, (0.2,), None, None),
    "d16_mixed_levels": (synth.GenSpec(L=4, H=2, d=16, S=700, seed=23, innov="t3", rho=(0.85, 0.99), n_outliers=1,
                                       outlier_scale=20.0), 128, 10, 127, (0.05, 0.1, 0.2, 0.4), None,
                         [3, 0, 2, 1, 1, 3]),
    "d32_escapes_R1": (synth.GenSpec(L=1, H=2, d=32, S=260, seed=24, innov="t3", rho=(0.9, 0.9), n_outliers=0),
                       64, 10, 1, (0.1,), None, None),
    "d64_escapes_R20": (synth.GenSpec(L=2, H=1, d=64, S=500, seed=25, innov="t3", rho=(0.85, 0.85), n_outliers=0),
                        250, 10, 20, (0.05,), None, None),
    "single_token": (synth.GenSpec(L=1, H=1, d=8, S=1, seed=26), 16, 10, 127, (0.1,), None, None),
    "group1_anchors_only": (synth.GenSpec(L=1, H=2, d=16, S=40, seed=27), 16, 1, 127, (0.1,), None, None),
    "chunk_shorter_than_group": (synth.GenSpec(L=1, H=1, d=8, S=23, seed=28), 4, 10, 127,
                                 (0.1,), None, None),
    "many_chunks_teams": (synth.GenSpec(L=1, H=1, d=128, S=2100, seed=29, innov="t3", rho=(0.85, 0.99)),
                          50, 10, 127, (0.1, 0.3), None, [i % 2 for i in range(42)]),
    # d = 128, 24 chunks of four levels, one level holding 21 of them
    "d128_levels_uneven": (synth.GenSpec(L=1, H=2, d=128, S=960, seed=30, innov="t3", rho=(0.85, 0.99),
                                                n_outliers=2, outlier_scale=20.0), 40, 10, 127,
                                  (0.05, 0.1, 0.2, 0.4), None, [0] * 21 + [1, 2, 3]),
    # separate K and V multipliers per layer (finer steps for keys)
    "d32_kv_asymmetric": (synth.GenSpec(L=3, H=2, d=32, S=400, seed=32, innov="t3", rho=(0.85, 0.99), n_outliers=1,
                                        outlier_scale=20.0), 128, 10, 127, (0.1,),
                          np.array([[0.25, 1.0], [0.5, 2.0], [1.0, 4.0]], np.float32), None),
    "d128_three_chunks_escapes_R3": (synth.GenSpec(L=1, H=1, d=128, S=300, seed=31, innov="t3", rho=(0.85, 0.9)),
                                100, 10, 3, (0.05,), None, None),
    # d = 128 with at most two chunks per (level, head): the thin-range
    # decoder (a team of four warps per stream); R = 3 makes escapes common,
    # so tokens whose words outrun the staging ring come up too
    "d128_thin_escapes_R3": (synth.GenSpec(L=1, H=2, d=128, S=200, seed=33, innov="t3", rho=(0.85, 0.9)),
                             100, 10, 3, (0.05,), None, None),
    # d = 128, six chunks of one level: k_dec128 with the u8 pair tables,
    # eight warps per CTA (MID); the last chunk is ragged
    "d128_mid_six_chunks": (synth.GenSpec(L=2, H=2, d=128, S=5 * 128 + 77, seed=35, innov="t3", rho=(0.85, 0.99),
                                          n_outliers=2, outlier_scale=20.0), 128, 10, 127, (0.05,), None, None),
    # eight chunks over four levels, two each; the last chunk is ragged
    "d128_thin_mixed_ragged": (synth.GenSpec(L=2, H=2, d=128, S=1000, seed=34, innov="t3", rho=(0.85, 0.99),
                                             n_outliers=2, outlier_scale=20.0), 128, 10, 127,
                               (0.05, 0.1, 0.2, 0.4), None, [0, 1, 2, 3, 3, 2, 1, 0]),
}


def _setup(orc, name):
    spec, C, G, R, lb, lm, lv = CASES[name]
    x = synth.generate(spec)
    cd = orc.Codec(spec.L, spec.H, spec.d, spec.S, C=C, G=G, R=R)
    cfg = cg.Config(spec.L, spec.H, spec.d, spec.S, C, G=G, R=R, level_base=lb, layer_mult=lm)
    levels = np.zeros(cd.n_chunks, np.uint8) if lv is None else np.asarray(lv, np.uint8)
    assert levels.size == cd.n_chunks
    return x, cd, cfg, levels, lb, lm


@pytest.mark.parametrize("name", list(CASES))
def test_fit_encode_decode_bit_exact(orc, name):
    x, cd, cfg, levels, lb, lm = _setup(orc, name)
    rc, tb_ref = orc.fit_tables(cd, list(lb), lm, x)
    assert rc == 0
    st, tb = gu.fit(cfg, x)
    assert st == cg.CG_OK
    assert tb.size == tb_ref.size
    if not np.array_equal(tb, tb_ref):
        bad = np.nonzero(tb != tb_ref)[0]
        pytest.fail(f"tables differ at {bad.size} bytes, first {bad[:8]}")
    rc, cont_ref, _ = orc.encode(cd, len(lb), tb_ref, x, levels)
    assert rc == 0
    st, cont, n = gu.encode(cfg, tb_ref, x, levels)
    assert st == cg.CG_OK and n == cont_ref.size
    if not np.array_equal(cont, cont_ref):
        bad = np.nonzero(cont != cont_ref)[0]
        pytest.fail(f"container differs at {bad.size} bytes, first {bad[:8]}")
    rc, y_ref = orc.decode(tb_ref, cont_ref)
    assert rc == 0
    st, y = gu.decode(cfg, tb_ref, cont_ref, fill=0x7E00)
    assert st == cg.CG_OK
    assert np.array_equal(y, y_ref)


def test_chunk_range_decode(orc):
    x, cd, cfg, levels, lb, lm = _setup(orc, "d16_mixed_levels")
    rc, tb = orc.fit_tables(cd, list(lb), lm, x)
    rc, cont, _ = orc.encode(cd, len(lb), tb, x, levels)
    _, full = orc.decode(tb, cont)
    for k0, k1 in ((0, 1), (2, 5), (5, 6), (3, 3)):
        st, y = gu.decode(cfg, tb, cont, k0, k1, fill=0x1234)
        assert st == cg.CG_OK
        t0, t1 = k0 * cd.C, min(k1 * cd.C, cd.S)
        assert np.array_equal(y[:, :, :, t0:t1], full[:, :, :, t0:t1])
        assert (y[:, :, :, :t0] == 0x1234).all() and (y[:, :, :, t1:] == 0x1234).all()


def test_chunk_range_decode_d128(orc):
    """Small chunk ranges at d = 128 (the thin-range decoder): each equals the
    oracle's decode of that range, and no other token is written."""
    x, cd, cfg, levels, lb, lm = _setup(orc, "d128_thin_mixed_ragged")
    rc, tb = orc.fit_tables(cd, list(lb), lm, x)
    rc, cont, _ = orc.encode(cd, len(lb), tb, x, levels)
    _, full = orc.decode(tb, cont)
    for k0, k1 in ((0, 1), (1, 3), (5, 8), (7, 8), (0, 8), (2, 2)):
        st, y = gu.decode(cfg, tb, cont, k0, k1, fill=0x1234)
        assert st == cg.CG_OK
        t0, t1 = k0 * cd.C, min(k1 * cd.C, cd.S)
        assert np.array_equal(y[:, :, :, t0:t1], full[:, :, :, t0:t1]), (k0, k1)
        assert (y[:, :, :, :t0] == 0x1234).all() and (y[:, :, :, t1:] == 0x1234).all()


def test_gpu_roundtrip_error_bound(orc):
    """GPU fit -> GPU encode -> GPU decode on a Llama-3-70B-like slice."""
    w = W.scaled(W.LLAMA3_70B, L=2, S=4608)
    x = synth.generate(w.gen)
    cfg = cg.Config.from_workload(w)
    st, tb = gu.fit(cfg, x)
    assert st == cg.CG_OK
    st, cont, n = gu.encode(cfg, tb, x, w.levels_for())
    assert st == cg.CG_OK
    st, y = gu.decode(cfg, tb, cont)
    assert st == cg.CG_OK
    cd = orc.Codec(w.L, w.H, w.d, w.S, w.C, w.G, w.R)
    rc, y_ref = orc.decode(tb, cont)
    assert rc == 0 and np.array_equal(y, y_ref)
    rc, tb_ref = orc.fit_tables(cd, list(w.level_base), None, x)
    assert rc == 0 and np.array_equal(tb, tb_ref)
    assert x.nbytes / cont.size > 2.0


# ---------------------------------------------------------------- failures
def _small(orc, name="d8_group7"):
    x, cd, cfg, levels, lb, lm = _setup(orc, name)
    rc, tb = orc.fit_tables(cd, list(lb), lm, x)
    rc, cont, _ = orc.encode(cd, len(lb), tb, x, levels)
    return x, cd, cfg, levels, tb, cont


# d = 8; d = 128 with 3 chunks (thin-range decoder); d = 128 with 42 chunks
# (a warp per stream, full tables); d = 128 with two chunks per level
# (thin-range decoder); d = 128 with six chunks (a warp per stream, u8 tables)
@pytest.mark.parametrize("name", ["d8_group7", "d128_ragged_chunks", "many_chunks_teams", "d128_thin_mixed_ragged",
                                  "d128_mid_six_chunks"])
def test_corrupt_containers_flagged(orc, name):
    x, cd, cfg, levels, tb, cont = _small(orc, name)
    assert gu.decode(cfg, tb, cont)[0] == cg.CG_OK
    bad = cont.copy()
    bad[0] ^= 1
    assert gu.decode(cfg, tb, bad)[0] == cg.CG_ERR_CORRUPT                     # magic
    assert gu.decode(cfg, tb, cont, nbytes=cont.size - 16)[0] == cg.CG_ERR_CORRUPT  # length
    base = int(cont[64:72].view(np.uint64)[0])
    nstr = cd.L * 2 * cd.H
    ng = -(-cd.C // cd.G)
    fixed_off = 16 + ((4 * nstr * cd.d + 15) // 16 * 16) + ((nstr * ng * cd.d + 15) // 16 * 16)
    offs = cont[base + fixed_off: base + fixed_off + 4 * nstr].view(np.uint32)
    for so in offs[:6]:
        sb = base + int(so)
        nw = int(cont[sb:sb + 4].view(np.uint32)[0])
        for pos in (sb + 16 + 1, sb + 16 + 4 * cd.d + 2 * (nw // 2)):
            b2 = cont.copy()
            b2[pos] ^= 0x20
            assert gu.decode(cfg, tb, b2)[0] == cg.CG_ERR_CORRUPT, pos
        b3 = cont.copy()
        b3[sb:sb + 4] = np.array([nw + 7], np.uint32).view(np.uint8)
        assert gu.decode(cfg, tb, b3)[0] == cg.CG_ERR_CORRUPT
    b4 = cont.copy()  # stream offset pointing outside its chunk
    b4[base + fixed_off: base + fixed_off + 4] = np.array([1 << 30], np.uint32).view(np.uint8)
    assert gu.decode(cfg, tb, b4)[0] == cg.CG_ERR_CORRUPT
    tb2 = tb.copy()  # a table whose CDF is not increasing
    _, _, cdfv = orc.tables_views(tb2, cd, len(CASES[name][4]))
    cdfv[0, 0, 0, 0, 100] = cdfv[0, 0, 0, 0, 99]
    assert gu.decode(cfg, tb2, cont)[0] == cg.CG_ERR_CORRUPT
    other = cg.Config(cd.L, cd.H, cd.d, cd.S, cd.C, G=cd.G + 1, R=cd.R, level_base=CASES[name][4])
    assert gu.decode(other, tb, cont)[0] == cg.CG_ERR_CORRUPT                  # dims mismatch


def test_nonfinite_flagged(orc):
    x, cd, cfg, levels, tb, cont = _small(orc)
    for bits in (0x7C00, 0xFC00, 0x7E01):
        for pos in ((0, 1, 2, 0, 3), (2, 0, 1, 5, 7)):  # an anchor and a delta token
            y = x.copy()
            y[pos] = bits
            assert gu.fit(cfg, y)[0] == cg.CG_ERR_NONFINITE
            assert gu.encode(cfg, tb, y, levels)[0] == cg.CG_ERR_NONFINITE


def test_capacity_flagged_and_size_reported(orc):
    x, cd, cfg, levels, tb, cont = _small(orc)
    st, out, n = gu.encode(cfg, tb, x, levels, cap=cont.size - 16)
    assert st == cg.CG_ERR_CAPACITY and n == cont.size
    st, out, n = gu.encode(cfg, tb, x, levels, cap=cont.size)
    assert st == cg.CG_OK and np.array_equal(out, cont)


def test_argument_errors_are_synchronous(orc):
    x, cd, cfg, levels, tb, cont = _small(orc)
    T = gu.torch()
    ws = cg.empty_u8(cg.cg_workspace_bytes(cfg, cg.CG_OP_DECODE))
    kv = T.zeros(x.size, dtype=T.int16, device="cuda")
    tbd, buf = gu.to_dev(tb), gu.to_dev(cont)
    assert cg.cg_decode(cfg, tbd, buf, cont.size, 0, cd.n_chunks + 1, kv, ws) == cg.CG_ERR_INVALID_ARG
    assert cg.cg_decode(cfg, tbd, buf, cont.size, 2, 1, kv, ws) == cg.CG_ERR_INVALID_ARG
    assert cg.cg_decode(cfg, tbd, buf[1:], cont.size - 1, 0, -1, kv, ws) == cg.CG_ERR_INVALID_ARG  # unaligned
    assert cg.cg_decode(cfg, tbd, buf, cont.size, 0, -1, kv, ws[:16]) == cg.CG_ERR_INVALID_ARG  # small ws
    assert cg.cg_encode(cfg, tbd, gu.to_dev(x), np.full(cd.n_chunks, 3, np.uint8), buf,
                        T.zeros(1, dtype=T.int64, device="cuda"),
                        cg.empty_u8(cg.cg_workspace_bytes(cfg, cg.CG_OP_ENCODE))) == cg.CG_ERR_INVALID_ARG


def _special_kv():
    """Constant channels, +-65504 extremes (reconstructions beyond the fp16
    range must clamp), subnormals and signed zeros."""
    f16 = lambda v: np.float16(v).view(np.uint16).item()  # noqa: E731
    L, H, d, S = 1, 1, 8, 60
    x = np.zeros((L, 2, H, S, d), np.uint16)
    x[..., 0] = f16(7.0)
    x[..., 1] = np.array([f16(65504), f16(-65504)] * 30)
    x[..., 2] = np.array([1, 0x8001, 3, 0x8000] * 15, np.uint16)
    x[..., 3] = f16(-0.0)
    x[..., 4] = np.array([f16(v) for v in np.linspace(-3, 3, S)])
    x[..., 5] = np.array(([f16(65504)] * 29 + [f16(-65504)]) * 2)
    x[..., 6] = np.array([f16(65504 - 32 * (t % 3)) for t in range(S)])
    x[..., 7] = np.array([f16(-65504 + 32 * (t % 5)) for t in range(S)])
    return x


@pytest.mark.parametrize("R,lb", [(127, (0.1,)), (127, (2.0,)), (3, (0.4,))])
def test_special_values_bit_exact(orc, R, lb):
    x = _special_kv()
    L, _, H, S, d = x.shape
    cd = orc.Codec(L, H, d, S, C=30, G=10, R=R)
    cfg = cg.Config(L, H, d, S, 30, G=10, R=R, level_base=lb)
    rc, tb_ref = orc.fit_tables(cd, list(lb), None, x)
    assert rc == 0
    st, tb = gu.fit(cfg, x)
    assert st == cg.CG_OK and np.array_equal(tb, tb_ref)
    rc, cont_ref, _ = orc.encode(cd, 1, tb_ref, x, np.zeros(cd.n_chunks, np.uint8))
    st, cont, n = gu.encode(cfg, tb_ref, x, np.zeros(cd.n_chunks, np.uint8))
    assert st == cg.CG_OK and np.array_equal(cont, cont_ref)
    rc, y_ref = orc.decode(tb_ref, cont_ref)
    st, y = gu.decode(cfg, tb_ref, cont_ref)
    assert rc == 0 and st == cg.CG_OK and np.array_equal(y, y_ref)
    assert (np.abs(y.view(np.float16).astype(np.float32)) <= 65504).all()


@pytest.mark.parametrize("name", ["tiny_workload", "d128_ragged_chunks", "d16_mixed_levels", "d64_escapes_R20",
                                  "d32_kv_asymmetric", "d128_three_chunks_escapes_R3"])
def test_entropy_bound_matches_oracle(orc, name):
    """cg_entropy_bound, from the fit's histograms, equals the oracle's
    entropy bound of a container with every chunk at that level: sum of n_s
    log2(N/n_s) per table / 8 + 4 bytes per escape + the structural bytes.
    The per-table logarithms are fp32 on the device, so the two agree to a
    few parts in 10^7."""
    spec, C, G, R, lb, lm, _ = CASES[name]
    x = synth.generate(spec)
    cfg = cg.Config(spec.L, spec.H, spec.d, spec.S, C=C, G=G, R=R, level_base=lb, layer_mult=lm)
    cd = orc.Codec(spec.L, spec.H, spec.d, spec.S, C=C, G=G, R=R)
    kvd = gu.to_dev(x)
    tb = cg.empty_u8(cg.cg_tables_bytes(cfg))
    ws = cg.empty_u8(cg.cg_workspace_bytes(cfg, cg.CG_OP_FIT))
    cg.check(cg.cg_fit_tables(cfg, kvd, tb, ws), "cg_fit_tables")
    gu.torch().cuda.synchronize()
    assert cg.cg_read_status(ws) == cg.CG_OK
    rc, tb_ref = orc.fit_tables(cd, list(lb), lm, x)
    assert rc == 0
    for lv in range(len(lb)):
        rc, cont, st = orc.encode(cd, len(lb), tb_ref, x, np.full(cd.n_chunks, lv, np.uint8))
        assert rc == 0
        want = orc.entropy_bound_bytes(st)
        got = cg.cg_entropy_bound(cfg, ws, lv)
        assert abs(got - want) <= 1e-6 * want, (lv, got, want)
        assert cont.size >= got * (1 - 1e-6)  # no container beats the bound
    if name == "d128_three_chunks_escapes_R3":
        assert st.n_esc > 0
    with pytest.raises(cg.CacheGenError):
        cg.cg_entropy_bound(cfg, ws, len(lb))
