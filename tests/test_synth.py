"""Sanity checks of the seeded input generator (not parity: its statistics)."""
import numpy as np

from kv_cache_compression_02_gb300 import synth
from kv_cache_compression_02_gb300 import workloads as W


def test_deterministic_and_addressable():
    spec = synth.GenSpec(L=2, H=3, d=8, S=50, seed=42, innov="t3", rho=(0.85, 0.99), n_outliers=2)
    a = synth.generate(spec, nthreads=1)
    b = synth.generate(spec, nthreads=5)
    assert np.array_equal(a, b)
    assert np.array_equal(synth.head(spec, 1, 0, 2), a[1, 0, 2])
    c = synth.generate(synth.GenSpec(L=2, H=3, d=8, S=50, seed=43, innov="t3", rho=(0.85, 0.99), n_outliers=2))
    assert not np.array_equal(a, c)


def test_moments():
    for innov in ("laplace", "t3"):
        spec = synth.GenSpec(L=1, H=1, d=16, S=20000, seed=7, innov=innov, rho=(0.9, 0.9), n_outliers=0)
        x = synth.head(spec, 0, 0, 0).view(np.float16).astype(np.float64)
        for j in range(16):
            rho, sc = synth.channel(spec, 0, 0, j)
            z = x[:, j] / sc
            assert abs(z.std() - 1.0) < 0.15
            r1 = np.corrcoef(z[:-1], z[1:])[0, 1]
            assert abs(r1 - 0.9) < 0.03


def test_outliers_and_levels():
    spec = W.LLAMA3_70B.gen
    n = 0
    for c in range(spec.H * spec.d):
        n += synth.channel(spec, 5, 1, c)[1] > 0  # touch every channel
    cnt = 0
    base = synth.GenSpec(L=spec.L, H=spec.H, d=spec.d, S=8, seed=spec.seed, innov=spec.innov, rho=spec.rho,
                         outlier_frac=0.0, outlier_scale=spec.outlier_scale)
    for c in range(spec.H * spec.d):
        cnt += abs(synth.channel(spec, 5, 1, c)[1] / synth.channel(base, 5, 1, c)[1] - 20.0) < 1e-9
    assert cnt == round(0.005 * spec.H * spec.d)
    lv = W.LONGCTX_MIXED.levels_for()
    assert lv.shape == (64,) and set(np.unique(lv)) <= {0, 1, 2, 3} and len(np.unique(lv)) == 4
