"""The five synthetic workloads the codec is tested and measured on.

Shapes follow the models the CacheGen pages evaluate on (Llama-7B,
Llama-3-8B, a Llama-3-70B geometry); the values come from the seeded
generator in :mod:`.synth`.  Each workload fixes the codec parameters:
chunk size C, anchor group G, level base steps and layer multipliers.

``chunk_levels`` says how chunks are assigned a compression level:
``"fixed"`` (level 0 everywhere), ``"each"`` (the whole context is encoded
once per level and each container is checked on its own) or ``"random"``
(one level per chunk drawn from the seed, as bandwidth-adaptive streaming
would pick them).
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

from .synth import GenSpec, chunk_levels as _draw_levels


@dataclass(frozen=True)
class Workload:
    name: str
    gen: GenSpec
    C: int
    G: int = 10
    R: int = 127
    level_base: tuple = (0.1,)
    layer_mult: tuple | None = None     # [L][2] or None: tiers 0.5/1/2 by thirds
    chunk_levels: str = "fixed"
    note: str = field(default="", compare=False)

    @property
    def L(self):
        return self.gen.L

    @property
    def H(self):
        return self.gen.H

    @property
    def d(self):
        return self.gen.d

    @property
    def S(self):
        return self.gen.S

    @property
    def n_chunks(self):
        return -(-self.S // self.C)

    @property
    def n_levels(self):
        return len(self.level_base)

    @property
    def elements(self):
        return self.L * 2 * self.H * self.S * self.d

    @property
    def fp16_bytes(self):
        return 2 * self.elements

    def levels_for(self, level: int = 0) -> np.ndarray:
        """Per-chunk levels (for "each", the container of one level)."""
        if self.chunk_levels == "random":
            return _draw_levels(self.gen.seed, self.n_chunks, self.n_levels)
        return np.full(self.n_chunks, level, np.uint8)

    def layer_mult_array(self):
        if self.layer_mult is None:
            return None
        return np.asarray(self.layer_mult, np.float32).reshape(self.L, 2)


TINY = Workload(
    "tiny_L2_H2_d64_S256",
    GenSpec(L=2, H=2, d=64, S=256, seed=0, innov="laplace", rho=(0.95, 0.95),
            outlier_scale=10.0, n_outliers=2),
    C=256, level_base=(0.1,), layer_mult=((0.5, 0.5), (2.0, 2.0)),
    note="one chunk, one level, m = 0.5 for layer 0 and 2 for layer 1")

LLAMA7B = Workload(
    "llama7b_L32_H32_d128_S4096",
    GenSpec(L=32, H=32, d=128, S=4096, seed=1, innov="laplace", rho=(0.95, 0.95),
            outlier_frac=0.01, outlier_scale=10.0),
    C=1024, level_base=(0.1,))

LLAMA3_8B = Workload(
    "llama3_8b_L32_H8_d128_S32768_3levels",
    GenSpec(L=32, H=8, d=128, S=32768, seed=2, innov="t3", rho=(0.85, 0.99),
            outlier_frac=0.01, outlier_scale=10.0),
    C=1536, level_base=(0.05, 0.1, 0.2), chunk_levels="each")

LLAMA3_70B = Workload(
    "llama3_70b_L80_H8_d128_S32768",
    GenSpec(L=80, H=8, d=128, S=32768, seed=3, innov="t3", rho=(0.85, 0.99),
            outlier_frac=0.005, outlier_scale=20.0),
    C=1536, level_base=(0.1,))

LONGCTX_MIXED = Workload(
    "llama3_70b_L80_H8_d128_S131072_mixed4",
    GenSpec(L=80, H=8, d=128, S=131072, seed=4, innov="t3", rho=(0.85, 0.99),
            outlier_frac=0.005, outlier_scale=20.0),
    C=2048, level_base=(0.05, 0.1, 0.2, 0.4), chunk_levels="random")

ALL = (TINY, LLAMA7B, LLAMA3_8B, LLAMA3_70B, LONGCTX_MIXED)
BY_NAME = {w.name: w for w in ALL}


def scaled(w: Workload, **kw) -> Workload:
    """The same generator and codec parameters at a different size."""
    g = w.gen
    gk = {k: kw.pop(k) for k in ("L", "H", "d", "S", "seed") if k in kw}
    gen = GenSpec(L=gk.get("L", g.L), H=gk.get("H", g.H), d=gk.get("d", g.d), S=gk.get("S", g.S),
                  seed=gk.get("seed", g.seed), innov=g.innov, rho=g.rho, outlier_frac=g.outlier_frac,
                  outlier_scale=g.outlier_scale, n_outliers=g.n_outliers)
    lm = kw.pop("layer_mult", None if gen.L != g.L else w.layer_mult)
    return Workload(kw.pop("name", w.name + "_scaled"), gen, C=kw.pop("C", w.C), G=kw.pop("G", w.G),
                    R=kw.pop("R", w.R), level_base=kw.pop("level_base", w.level_base), layer_mult=lm,
                    chunk_levels=kw.pop("chunk_levels", w.chunk_levels))
