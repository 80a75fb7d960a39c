"""Pins of the CPU oracle against facts fixed outside the oracle itself.

Each test names what it checks against: IEEE/numpy conversions, closed
forms, textbook routines, brute force on tiny inputs, invariants, or the
hand-worked byte fixtures under tests/golden/.  A plausible slip in the
oracle (a dropped term, a sign, an index, a transposed operand, a reversed
word order) fails at least one of them.
"""
import itertools
import math
from fractions import Fraction

import numpy as np
import pytest

from kv_cache_compression_02_gb300 import synth
from kv_cache_compression_02_gb300 import workloads as W
from tests.golden.load import load as load_golden

F16_FINITE = np.array([b for b in range(65536) if (b >> 10) & 31 != 31], np.uint16)


def f16(v):
    return np.float16(v).view(np.uint16).item()


def fp16_ulp(v16: np.ndarray) -> np.ndarray:
    """Spacing of fp16 numbers at each value (2^-24 in the subnormal range)."""
    a = np.abs(v16.astype(np.float64))
    e = np.floor(np.log2(np.maximum(a, 2.0 ** -14)))
    return 2.0 ** (e - 10)


# ---------------------------------------------------------------- binary16
def test_f16_to_f32_exhaustive_vs_numpy(orc):
    bits = np.arange(65536, dtype=np.uint16)
    ref = bits.view(np.float16).astype(np.float32)
    got = np.array([orc.f16_to_f32(int(b)) for b in bits], np.float32)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan].view(np.uint32), ref[~nan].view(np.uint32))


def test_f32_to_f16_rn_vs_numpy(orc):
    fin = F16_FINITE.view(np.float16).astype(np.float32)
    pos = np.sort(fin[fin > 0])
    mids = ((pos[:-1].astype(np.float64) + pos[1:]) / 2).astype(np.float32)  # exact ties
    rng = np.random.default_rng(7)
    rnd = (rng.standard_normal(20000) * np.exp(rng.uniform(-20, 11, 20000))).astype(np.float32)
    extra = np.array([0.0, -0.0, 65504, 65519.99, 65520, 70000, -65520, 2 ** -25, 2 ** -24 * 1.5,
                      np.inf, -np.inf], np.float32)
    xs = np.concatenate([fin, mids, -mids, rnd, extra])
    with np.errstate(over="ignore"):  # values past the fp16 range round to infinity, as intended
        ref = xs.astype(np.float16).view(np.uint16)
    got = np.array([orc.f32_to_f16(float(v)) for v in xs], np.uint16)
    assert np.array_equal(got, ref)


# ---------------------------------------------------------------- sigma
def test_sigma_closed_forms(orc):
    assert orc.channel_sigma(np.full(37, f16(3.25), np.uint16)) == 0.0
    for a in (0.5, 1.0, 3.0, 1000.0, 2.0 ** -20, 65504.0):
        x = np.array([f16(a), f16(-a)] * 50, np.uint16)
        assert orc.channel_sigma(x) == np.float32(np.float16(a))
    # two values with equal counts: sigma = |a - b| / 2
    for a, b in ((1.0, 2.0), (-7.5, 3.25), (100.0, 101.0)):
        x = np.array([f16(a)] * 21 + [f16(b)] * 21, np.uint16)
        assert orc.channel_sigma(x) == np.float32(abs(a - b) / 2)


def test_sigma_vs_numpy_and_exact(orc):
    rng = np.random.default_rng(3)
    for trial in range(40):
        n = int(rng.integers(1, 3000))
        scale = float(np.exp(rng.uniform(-12, 9)))
        v = (rng.standard_normal(n) * scale + rng.standard_normal() * scale * 3).astype(np.float16)
        v = np.clip(v, -65504, 65504).astype(np.float16)
        got = orc.channel_sigma(v.view(np.uint16))
        ref = np.float32(np.std(v.astype(np.float64)))
        assert abs(float(got) - float(ref)) <= float(np.spacing(np.float32(ref))) + 1e-45
        # exact rational variance, independent of any floating-point order
        fr = [Fraction(float(t)) for t in v]
        mu = sum(fr) / n
        var = sum((t - mu) ** 2 for t in fr) / n
        exact = math.sqrt(float(var))
        assert abs(float(got) - exact) <= 1.01 * float(np.spacing(np.float32(exact))) + 1e-45


# ---------------------------------------------------------------- step
def test_step_floor_and_values(orc):
    s, r = orc.step(0.1, 1.0, 0.0)
    assert s == np.float32(2.0 ** -12) and r == np.float32(4096.0)
    s, r = orc.step(0.5, 2.0, 3.0)
    assert s == 3.0 and r == np.float32(1 / 3)
    s, r = orc.step(0.25, 0.5, 8.0)
    assert s == 1.0 and r == 1.0
    # layer-adaptive: larger multiplier never gives a finer step
    assert orc.step(0.1, 0.5, 2.0)[0] < orc.step(0.1, 1.0, 2.0)[0] < orc.step(0.1, 2.0, 2.0)[0]


# ---------------------------------------------------------------- anchors
def test_anchor_scale_and_code(orc):
    s, inv = orc.anchor_scale(0.0)
    assert s == 0 and inv == 0
    q, ah = orc.anchor_code(5.0, s, inv)
    assert q == 0 and ah == 0.0
    s, inv = orc.anchor_scale(127.0)
    assert s == 1.0 and inv == 1.0
    assert orc.anchor_code(-127.0, s, inv) == (-127, -127.0)
    assert orc.anchor_code(2.5, s, inv)[0] == 2      # ties to even
    assert orc.anchor_code(3.5, s, inv)[0] == 4
    assert orc.anchor_code(-2.5, s, inv)[0] == -2


def test_group1_is_textbook_int8_absmax(orc):
    """G = 1: every token is an anchor, so the codec must equal per-chunk,
    per-channel symmetric int8 absmax quantization, restated independently."""
    spec = synth.GenSpec(L=2, H=2, d=16, S=37, seed=11, innov="t3", rho=(0.9, 0.9),
                         n_outliers=1, outlier_scale=10.0)
    x = synth.generate(spec)
    cd = orc.Codec(2, 2, 16, 37, C=16, G=1)
    rc, tb = orc.fit_tables(cd, [0.1], None, x)
    assert rc == 0
    rc, cont, st = orc.encode(cd, 1, tb, x, np.zeros(cd.n_chunks, np.uint8))
    assert rc == 0 and st.n_symbols == 0
    rc, y = orc.decode(tb, cont)
    assert rc == 0
    xf = x.view(np.float16).astype(np.float32)
    ref = np.empty_like(xf)
    for k in range(cd.n_chunks):
        blk = xf[:, :, :, k * 16:(k + 1) * 16, :]
        amax = np.abs(blk).max(axis=3, keepdims=True)
        with np.errstate(divide="ignore", invalid="ignore"):
            scale = np.where(amax > 0, amax / np.float32(127), 0).astype(np.float32)
            inv = np.where(amax > 0, np.float32(127) / amax, 0).astype(np.float32)
        qq = np.clip(np.rint(blk * inv), -127, 127).astype(np.int8).astype(np.float32)  # int8 code
        ref[:, :, :, k * 16:(k + 1) * 16, :] = qq * scale
    assert np.array_equal(y, ref.astype(np.float16).view(np.uint16))


# ---------------------------------------------------------------- deltas: error bound
@pytest.mark.parametrize("ahat,step_", [(0.0, 0.1), (1.984375, 0.25), (-3.1, 2.0 ** -12),
                                        (1000.0, 37.5), (-60000.0, 900.0)])
def test_delta_error_bound_exhaustive(orc, ahat, step_):
    """For every finite fp16 x: |fp16(x_hat) - x| <= step/2 plus the fp32
    rounding of the quantizer and of the fma, plus half an fp16 ulp."""
    ahat = np.float32(ahat)
    st, rp = np.float32(step_), np.float32(1.0) / np.float32(step_)
    xs = F16_FINITE[::3]
    xv = xs.view(np.float16).astype(np.float64)
    out = np.array([orc.reconstruct(orc.delta_code(float(v), ahat, rp), st, ahat) for v in xv], np.uint16)
    y = out.view(np.float16).astype(np.float64)
    bound = (float(st) / 2 + np.abs(xv - float(ahat)) * 2.0 ** -21 + np.abs(xv) * 2.0 ** -23
             + fp16_ulp(out.view(np.float16)) / 2)
    assert np.all(np.abs(y - xv) <= bound)


def test_symbols_and_escape(orc):
    assert orc.symbol(0) == 127 and orc.symbol(-127) == 0 and orc.symbol(127) == 254
    assert orc.symbol(128) == 255 and orc.symbol(-128) == 255
    assert orc.symbol(2, R=1) == 255 and orc.symbol(-1, R=1) == 126


# ---------------------------------------------------------------- normalisation
def test_normalize_invariants(orc):
    rng = np.random.default_rng(5)
    cases = [np.zeros(256, np.int64), np.ones(256, np.int64), np.eye(256, dtype=np.int64)[3] * 10 ** 9]
    for _ in range(60):
        n = np.zeros(256, np.int64)
        k = int(rng.integers(1, 256))
        idx = rng.choice(256, k, replace=False)
        n[idx] = rng.geometric(rng.uniform(1e-4, 0.5), k)
        cases.append(n)
    tie = np.zeros(256, np.int64)
    tie[[40, 41, 200]] = (7, 7, 5)   # remainder 2 goes to symbol 40
    cases.append(tie)
    for n in cases:
        f, c = orc.normalize(n)
        N = int(n.sum())
        assert int(f.sum()) == 65536 and f.min() >= 1
        assert c[0] == 0 and np.array_equal(np.diff(c.astype(np.int64)), f.astype(np.int64))
        arg = 127 if N == 0 else int(np.argmax(n))      # argmax: lowest index on ties
        for s in range(256 if N else 0):
            dev = int(f[s]) - n[s] * 65536 / N
            if s == arg:
                assert -256 * n[s] / max(N, 1) - 1e-9 <= dev <= 257
            else:
                assert abs(dev) <= 1 + 256 * n[s] / max(N, 1) + 1e-9
        if N == 0:
            assert f[127] == 65536 - 255
    f, _ = orc.normalize(tie)
    assert f[40] > f[41]                                # remainder went to the lowest index


# ---------------------------------------------------------------- rANS
def _tables_for(freqs_by_lane):
    d = len(freqs_by_lane)
    f = np.ones((d, 256), np.uint32)
    for j, fj in enumerate(freqs_by_lane):
        for s, v in fj.items():
            f[j, s] = v
        f[j, 127] += 65536 - f[j].sum()
    cdf = np.zeros((d, 257), np.uint32)
    cdf[:, 1:] = np.cumsum(f, axis=1)
    return f, cdf


def _ans_bigint(seq, f, cdf):
    """Unbounded-precision ANS (no renormalisation): x <- floor(x/f)M + x mod f + cdf."""
    x = 1 << 16
    for s in reversed(seq):
        x = (x // int(f[s])) * 65536 + x % int(f[s]) + int(cdf[s])
    return x


def test_rans_bruteforce_roundtrip(orc):
    tables = [
        [{126: 100, 128: 30000}],                         # skewed, 127 takes the rest
        [{126: 1, 128: 1}],                               # two rarest possible symbols
        [{126: 20000, 128: 20000, 255: 5}],               # with the escape symbol
        [{126: 3, 128: 60000}, {126: 32768, 128: 16384}],  # two lanes, different tables
    ]
    alph = [126, 127, 128, 255]
    for tab in tables:
        f, cdf = _tables_for(tab)
        d = len(tab)
        for n in range(0, 5):
            for seq in itertools.product(alph, repeat=n * d):
                sym = np.array(seq, np.uint8).reshape(n, d)
                q = sym.astype(np.int32) - 127
                q[sym == 255] = -1000 - np.arange((sym == 255).sum())
                st, w = orc.rans_encode(sym, q, f, cdf)
                rc, s2, q2 = orc.rans_decode(n, st, w, int((sym == 255).sum()), f, cdf)
                assert rc == 0
                assert np.array_equal(s2, sym) and np.array_equal(q2, q)


def test_rans_state_matches_unbounded_ans(orc):
    """Without renormalisation the 32-bit coder must equal plain ANS."""
    f, cdf = _tables_for([{120: 4000, 130: 9000}])
    rng = np.random.default_rng(2)
    for _ in range(50):
        seq = list(rng.choice([120, 127, 130], size=int(rng.integers(1, 3))))
        ref = _ans_bigint(seq, f[0], cdf[0])
        sym = np.array(seq, np.uint8).reshape(-1, 1)
        st, w = orc.rans_encode(sym, sym.astype(np.int32) - 127, f, cdf)
        if ref < 2 ** 32:
            assert len(w) == 0 and int(st[0]) == ref


def test_rans_code_length(orc):
    rng = np.random.default_rng(9)
    for d in (1, 3, 8):
        n = 4000
        p = rng.dirichlet(np.ones(12) * 0.7)
        syms = rng.choice(np.arange(120, 132), size=(n, d), p=p).astype(np.uint8)
        counts = [np.bincount(syms[:, j], minlength=256) for j in range(d)]
        f = np.zeros((d, 256), np.uint32)
        cdf = np.zeros((d, 257), np.uint32)
        for j in range(d):
            f[j], cdf[j] = orc.normalize(counts[j])
        st, w = orc.rans_encode(syms, syms.astype(np.int32) - 127, f, cdf)
        ideal = sum(-np.log2(f[j][syms[:, j]] / 65536.0).sum() for j in range(d))
        bits = 16 * len(w)
        assert ideal - 16 * d <= bits <= ideal + 16 * d
        rc, s2, _ = orc.rans_decode(n, st, w, 0, f, cdf)
        assert rc == 0 and np.array_equal(s2, syms)


# ---------------------------------------------------------------- hand-worked bytes
def _hand_kv():
    v = [f16(127 / 64), f16(63 / 64), f16(127 / 64), f16(63 / 64)]
    return np.array(v * 2, np.uint16).reshape(1, 2, 1, 4, 1)


@pytest.mark.parametrize("fixture,R", [("hand_worked_L1_H1_d1_S4.txt", 127), ("hand_worked_escape_R1.txt", 1)])
def test_hand_worked_golden(orc, fixture, R):
    g = load_golden(fixture)
    cd = orc.Codec(1, 1, 1, 4, C=4, G=2, R=R)
    kv = _hand_kv()
    rc, tb = orc.fit_tables(cd, [0.5], np.ones((1, 2), np.float32), kv)
    assert rc == 0 and tb.size == 1120
    head = g["tables_head"]
    assert np.array_equal(tb[:head.size], head)
    _, _, cdf = orc.tables_views(tb, cd, 1)
    expect = np.arange(256) + np.where(np.arange(256) > 123, 65280, 0) if R == 127 else np.arange(256)
    assert np.array_equal(cdf[0, 0, 0, 0], expect) and np.array_equal(cdf[0, 0, 1, 0], expect)
    rc, cont, st = orc.encode(cd, 1, tb, kv, [0])
    assert rc == 0
    assert np.array_equal(cont, g["container"])
    rc, y = orc.decode(tb, cont)
    assert rc == 0 and np.array_equal(y, kv)


# ---------------------------------------------------------------- whole codec
def _roundtrip(orc, spec, C, G, R=127, levels=(0.1,), mult=None, chunk_levels=None):
    x = synth.generate(spec)
    cd = orc.Codec(spec.L, spec.H, spec.d, spec.S, C=C, G=G, R=R)
    rc, tb = orc.fit_tables(cd, list(levels), mult, x)
    assert rc == 0
    lv = np.zeros(cd.n_chunks, np.uint8) if chunk_levels is None else np.asarray(chunk_levels, np.uint8)
    rc, cont, st = orc.encode(cd, len(levels), tb, x, lv)
    assert rc == 0
    rc, y = orc.decode(tb, cont)
    assert rc == 0
    return x, y, tb, cont, st, cd, lv


def _check_error_bound(orc, x, y, tb, cd, lv, nl):
    """Per element: deltas within step/2 (+fp32 and fp16 rounding), anchors
    within s/2 (+ rounding)."""
    step_, _, _ = orc.tables_views(tb, cd, nl)
    xf = x.view(np.float16).astype(np.float64)
    yf = y.view(np.float16).astype(np.float64)
    err = np.abs(xf - yf)
    L, _, H, S, d = x.shape
    for k in range(cd.n_chunks):
        t0, t1 = k * cd.C, min((k + 1) * cd.C, S)
        st = step_[lv[k]].reshape(L, 2, H, 1, d).astype(np.float64)
        blk = slice(t0, t1)
        rel = np.arange(t1 - t0)
        anchor = (rel % cd.G) == 0
        amax = np.abs(xf[:, :, :, blk][:, :, :, anchor]).max(axis=3, keepdims=True)
        sa = amax / 127
        e = err[:, :, :, blk]
        ul = fp16_ulp(y[:, :, :, blk].view(np.float16)) / 2
        xa = np.abs(xf[:, :, :, blk])
        ba = sa / 2 * (1 + 2.0 ** -20) + ul + xa * 2.0 ** -22
        bd = st / 2 + (xa + amax) * 2.0 ** -21 + xa * 2.0 ** -23 + sa / 2 * 0 + ul
        assert np.all(e[:, :, :, anchor] <= ba[:, :, :, anchor])
        assert np.all(e[:, :, :, ~anchor] <= bd[:, :, :, ~anchor])


def test_tiny_workload_roundtrip_and_bound(orc):
    w = W.TINY
    x, y, tb, cont, st, cd, lv = _roundtrip(orc, w.gen, w.C, w.G, levels=w.level_base,
                                            mult=w.layer_mult_array())
    _check_error_bound(orc, x, y, tb, cd, lv, 1)
    assert x.nbytes / cont.size > 2.5


def test_ratio_within_one_percent_of_entropy_bound(orc):
    spec = W.scaled(W.LLAMA3_70B, L=2, H=2, S=8192).gen
    x, y, tb, cont, st, cd, lv = _roundtrip(orc, spec, C=2048, G=10)
    bound = orc.entropy_bound_bytes(st)
    assert cont.size <= 1.01 * bound
    assert cont.size >= bound            # the coder cannot beat the empirical entropy here
    # the split of the container adds up
    assert st.fixed_bytes + st.state_bytes + 2 * st.n_words + st.pad_bytes == cont.size


@pytest.mark.parametrize("S,C,G,d", [(1, 4, 10, 8), (11, 11, 10, 2), (23, 15, 10, 1), (40, 7, 3, 8),
                                     (64, 64, 64, 4), (10, 3, 10, 2)])
def test_ragged_shapes(orc, S, C, G, d):
    spec = synth.GenSpec(L=1, H=2, d=d, S=S, seed=S * 7 + d, innov="t3", rho=(0.85, 0.99), n_outliers=0)
    x, y, tb, cont, st, cd, lv = _roundtrip(orc, spec, C=C, G=G)
    _check_error_bound(orc, x, y, tb, cd, lv, 1)


def test_forced_escapes_roundtrip(orc):
    spec = synth.GenSpec(L=1, H=1, d=8, S=200, seed=5, innov="t3", rho=(0.9, 0.9), n_outliers=0)
    x, y, tb, cont, st, cd, lv = _roundtrip(orc, spec, C=64, G=10, R=1)
    assert st.n_esc > 100
    _check_error_bound(orc, x, y, tb, cd, lv, 1)


def test_mixed_levels_roundtrip(orc):
    spec = synth.GenSpec(L=3, H=1, d=8, S=300, seed=8, innov="t3", rho=(0.85, 0.99), n_outliers=1,
                         outlier_scale=20.0)
    lv = [0, 3, 1, 2, 3]
    x, y, tb, cont, st, cd, lvv = _roundtrip(orc, spec, C=64, G=10, levels=(0.05, 0.1, 0.2, 0.4),
                                             chunk_levels=lv)
    _check_error_bound(orc, x, y, tb, cd, lvv, 4)
    # decode of a sub-range only touches that range
    rc, part = orc.decode(tb, cont, 1, 3)
    assert rc == 0
    assert np.array_equal(part[:, :, :, 64:192], y[:, :, :, 64:192])
    assert not part[:, :, :, :64].any() and not part[:, :, :, 192:].any()


def test_special_values(orc):
    L, H, d, S = 1, 1, 8, 30
    x = np.zeros((L, 2, H, S, d), np.uint16)
    x[..., 0] = f16(7.0)                                   # constant channel: sigma 0
    x[..., 1] = np.array([f16(65504), f16(-65504)] * 15)   # extremes
    x[..., 2] = np.array([1, 0x8001, 3, 0x8000] * 7 + [0, 0], np.uint16)  # subnormals, -0
    x[..., 3] = f16(-0.0)
    x[..., 4] = np.array([f16(v) for v in np.linspace(-3, 3, S)])
    x[..., 5] = np.array([f16(65504)] * 29 + [f16(-65504)])
    cd = orc.Codec(L, H, d, S, C=S, G=10)
    rc, tb = orc.fit_tables(cd, [0.1], None, x)
    assert rc == 0
    step_, recip, _ = orc.tables_views(tb, cd, 1)
    assert step_[0, 0, 0, 0] == np.float32(2.0 ** -12)
    rc, cont, st = orc.encode(cd, 1, tb, x, [0])
    assert rc == 0
    rc, y = orc.decode(tb, cont)
    assert rc == 0
    _check_error_bound(orc, x, y, tb, cd, np.zeros(1, np.uint8), 1)
    assert np.array_equal(y[..., 0], x[..., 0])


def test_nonfinite_rejected(orc):
    cd = orc.Codec(1, 1, 4, 20, C=20, G=10)
    x = np.zeros((1, 2, 1, 20, 4), np.uint16)
    x[0, 1, 0, 13, 2] = 0x7C00   # +Inf
    rc, tb = orc.fit_tables(cd, [0.1], None, x)
    assert rc == orc.ERR_NONFINITE
    x[0, 1, 0, 13, 2] = 0x7E01   # NaN
    rc, tb = orc.fit_tables(cd, [0.1], None, x)
    assert rc == orc.ERR_NONFINITE
    good = np.zeros_like(x)
    rc, tb = orc.fit_tables(cd, [0.1], None, good)
    rc, cont, st = orc.encode(cd, 1, tb, x, [0])
    assert rc == orc.ERR_NONFINITE


def test_corrupt_containers_rejected(orc):
    spec = synth.GenSpec(L=1, H=2, d=8, S=100, seed=3, innov="laplace", rho=(0.95, 0.95), n_outliers=0)
    x, y, tb, cont, st, cd, lv = _roundtrip(orc, spec, C=50, G=10)
    bad = cont.copy()
    bad[0] ^= 1
    assert orc.decode(tb, bad)[0] == orc.ERR_CORRUPT             # magic
    assert orc.decode(tb, cont[:-16])[0] == orc.ERR_CORRUPT      # truncated
    # flip a bit of a lane state and of a word in every stream, one at a time
    base = int(cont[64:72].view(np.uint64)[0])
    nstr = 4
    ng = 5
    fixed = 16 + 4 * nstr * 8 + ((nstr * ng * 8 + 15) & ~15) + 16
    offs = cont[base + fixed - 16: base + fixed].view(np.uint32)
    for so in offs:
        sb = base + int(so)
        nw = int(cont[sb:sb + 4].view(np.uint32)[0])
        for pos in (sb + 16 + 5, sb + 16 + 32 + 1, sb + 16 + 32 + 2 * (nw // 2)):
            b2 = cont.copy()
            b2[pos] ^= 0x10
            assert orc.decode(tb, b2)[0] == orc.ERR_CORRUPT, pos
        b3 = cont.copy()
        b3[sb:sb + 4] = np.array([nw + 1], np.uint32).view(np.uint8)
        assert orc.decode(tb, b3)[0] == orc.ERR_CORRUPT


def test_capacity_reported(orc):
    import ctypes
    spec = synth.GenSpec(L=1, H=1, d=8, S=64, seed=1, n_outliers=0)
    x = synth.generate(spec)
    cd = orc.Codec(1, 1, 8, 64, C=64, G=10)
    rc, tb = orc.fit_tables(cd, [0.1], None, x)
    out = np.zeros(200, np.uint8)
    nb = ctypes.c_uint64(0)
    lv = np.zeros(1, np.uint8)
    rc = orc.lib().orc_encode(orc._ref(cd.dims()), 1, orc._p(tb), orc._p(x), orc._p(lv), orc._p(out), 200,
                              orc._ref(nb), None)
    assert rc == orc.ERR_CAPACITY


def test_hand_worked_interleaved_renorm(orc):
    """Fixes the word order of interleaved lanes: pushes reversed, token
    ascending then lane ascending."""
    g = load_golden("hand_worked_rans_d2.txt")
    f, cdf = _tables_for([{}, {}])
    sym = np.array([[0, 127], [127, 254]], np.uint8)
    st, w = orc.rans_encode(sym, sym.astype(np.int32) - 127, f, cdf)
    assert np.array_equal(st.view(np.uint8), g["states"])
    assert np.array_equal(w.view(np.uint8), g["words"])
    rc, s2, _ = orc.rans_decode(2, st, w, 0, f, cdf)
    assert rc == 0 and np.array_equal(s2, sym)


def test_paged_layout_hand_example(orc):
    """The block-table layout (pools [L][2][n_blocks][H][bt][d]) on a case
    worked by hand: S=5 tokens in blocks of 2, table [2, 0, 1]."""
    L, H, S, d = 1, 2, 5, 2
    kv = np.zeros((L, 2, H, S, d), np.uint16)
    for k in range(2):
        for h in range(H):
            for t in range(S):
                for j in range(d):
                    kv[0, k, h, t, j] = 1000 * k + 100 * h + 10 * t + j + 1
    pools = orc.paged_from_contiguous(kv, [2, 0, 1], 2, 3, fill=7)
    assert pools.shape == (1, 2, 3, 2, 2, 2)
    assert pools[0, 1, 0, 1, 1, 0] == 1131    # V, block 0 row 1 = token 3, head 1, j 0
    assert pools[0, 0, 2, 1, 0, 1] == 102     # K, block 2 row 0 = token 0, head 1, j 1
    assert pools[0, 0, 1, 0, 0, 0] == 41      # block 1 row 0 = token 4
    assert (pools[0, :, 1, :, 1, :] == 7).all()  # block 1 row 1: no token (S = 5)
    # only the listed tokens are placed
    part = orc.paged_from_contiguous(kv, [2, 0, 1], 2, 3, fill=0, tokens=[2, 3])
    assert (part[0, :, 2] == 0).all() and (part[0, :, 1] == 0).all()
    assert part[0, 0, 0, 0, 0, 0] == 21 and part[0, 0, 0, 0, 1, 0] == 31


def test_kv_asymmetric_multipliers(orc):
    """Separate K and V multipliers per layer (Guide to CacheGen, pillar 1:
    keys need finer steps than values): with the same data in K and V, a
    channel's V step over its K step is the multiplier ratio, exactly for a
    power-of-two ratio; every table is otherwise what one multiplier gives."""
    spec = synth.GenSpec(L=2, H=1, d=8, S=200, seed=71, innov="laplace", rho=(0.9, 0.9), n_outliers=0)
    x = synth.generate(spec)
    x[:, 1] = x[:, 0]  # V = K
    cd = orc.Codec(2, 1, 8, 200, C=100, G=10)
    lm = np.array([[0.25, 1.0], [0.5, 2.0]], np.float32)  # V steps 4x the K steps
    rc, tb = orc.fit_tables(cd, [0.1], lm, x)
    assert rc == 0
    step_, recip, cdf = orc.tables_views(tb, cd, 1)
    for l in range(2):
        big = step_[0, l, 0] > 2.0 ** -12 * 4  # away from the step floor
        assert np.array_equal(step_[0, l, 1][big], 4 * step_[0, l, 0][big])
    # K of layer 0 equals a fit with that multiplier for both K and V
    rc, tb_k = orc.fit_tables(cd, [0.1], np.array([[0.25, 0.25], [0.5, 0.5]], np.float32), x)
    s_k, _, c_k = orc.tables_views(tb_k, cd, 1)
    assert np.array_equal(s_k[0, :, 0], step_[0, :, 0]) and np.array_equal(c_k[0, :, 0], cdf[0, :, 0])
    cont_rc, cont, _ = orc.encode(cd, 1, tb, x, np.zeros(cd.n_chunks, np.uint8))
    rc, y = orc.decode(tb, cont)
    assert cont_rc == 0 and rc == 0
    err = np.abs(y.view(np.float16).astype(np.float64) - x.view(np.float16).astype(np.float64))
    assert err[:, 0].max() < err[:, 1].max()  # finer K steps, smaller K error


def test_outlier_channel_does_not_touch_other_channels(orc):
    """Outlier channels are kept from corrupting the regular channels'
    distributions (Guide to CacheGen, pillar 3: the sparse outlier table).
    Here every channel has its own step and frequency table, so scaling one
    channel by 20x leaves every other channel's table and decoded values
    unchanged."""
    spec = synth.GenSpec(L=1, H=2, d=16, S=300, seed=72, innov="t3", rho=(0.9, 0.9), n_outliers=0)
    x = synth.generate(spec)
    y = x.copy()
    ch = y[0, 0, 1, :, 5].view(np.float16).astype(np.float32) * 20
    y[0, 0, 1, :, 5] = ch.astype(np.float16).view(np.uint16)
    cd = orc.Codec(1, 2, 16, 300, C=100, G=10)
    rc, tx = orc.fit_tables(cd, [0.1], None, x)
    rc2, ty = orc.fit_tables(cd, [0.1], None, y)
    assert rc == rc2 == 0
    sx, _, cx = orc.tables_views(tx, cd, 1)
    sy, _, cy = orc.tables_views(ty, cd, 1)
    other = np.ones(2 * 16, bool)
    other[16 + 5] = False  # head 1, channel 5 of K
    assert np.array_equal(sx[0, 0, 0][other], sy[0, 0, 0][other])
    assert np.array_equal(cx[0, 0, 0][other], cy[0, 0, 0][other])
    assert not np.array_equal(sx[0, 0, 0][~other], sy[0, 0, 0][~other])
    dx = orc.decode(tx, orc.encode(cd, 1, tx, x, np.zeros(3, np.uint8))[1])[1]
    dy = orc.decode(ty, orc.encode(cd, 1, ty, y, np.zeros(3, np.uint8))[1])[1]
    mask = np.ones(dx.shape, bool)
    mask[0, 0, 1, :, 5] = False
    assert np.array_equal(dx[mask], dy[mask])


def test_table_entropy_closed_forms(orc):
    """sum_s n_s log2(N / n_s): uniform counts give N log2(k); two symbols
    split p, 1-p give N H2(p); an empty or one-symbol table carries 0 bits."""
    n = np.zeros(256, np.uint64)
    assert orc.table_entropy(n) == 0.0
    n[127] = 1000
    assert orc.table_entropy(n) == 0.0
    n[:] = 0
    n[:16] = 5
    assert abs(orc.table_entropy(n) - 80 * 4.0) < 1e-9
    n[:] = 0
    n[3], n[250] = 1, 3
    h2 = -(0.25 * np.log2(0.25) + 0.75 * np.log2(0.75))
    assert abs(orc.table_entropy(n) - 4 * h2) < 1e-12


def test_per_stream_accounting_adds_up_to_the_container(orc):
    """Encoding stream by stream with the per-table symbol counts and the
    size split reproduces orc_encode's statistics of the whole container: the
    entropy term (summed per table), escapes, words, flush and the structural
    bytes (container part plus 16 per stream).  This is how the full-size
    parity pass bounds the GPU's containers stream by stream."""
    spec = synth.GenSpec(L=2, H=2, d=16, S=700, seed=3, innov="t3", rho=(0.85, 0.99), n_outliers=1,
                         outlier_scale=20.0)
    levels, chunk_levels = (0.05, 0.2), [0, 1, 1, 0, 1, 0]
    x, y, tb, cont, st, cd, lv = _roundtrip(orc, spec, C=128, G=10, levels=levels, chunk_levels=chunk_levels,
                                            R=20)
    step_, recip, cdf = orc.tables_views(tb, cd, len(levels))
    acc = orc.Stats()
    h = 0.0
    nstr = spec.L * 2 * spec.H
    for si in range(nstr):
        l, kv, hh = si // (2 * spec.H), (si // spec.H) % 2, si % spec.H
        c0 = hh * spec.d
        counts = np.zeros((len(levels), spec.d, 256), np.uint64)
        for k in range(cd.n_chunks):
            v = lv[k]
            n, blk, s, anc = orc.encode_stream(cd, x[l, kv, hh], k, step_[v, l, kv, c0:c0 + spec.d],
                                               recip[v, l, kv, c0:c0 + spec.d], cdf[v, l, kv, c0:c0 + spec.d],
                                               symcount=counts[v], stats=acc)
            assert n > 0
        h += sum(orc.table_entropy(counts[v, j]) for v in range(len(levels)) for j in range(spec.d))
    assert acc.n_esc == st.n_esc and acc.n_esc > 0
    assert acc.n_words == st.n_words and acc.n_symbols == st.n_symbols and acc.state_bytes == st.state_bytes
    assert acc.fixed_bytes + orc.container_fixed_bytes(cd) == st.fixed_bytes
    assert abs(h - st.entropy_bits) <= 1e-9 * st.entropy_bits
