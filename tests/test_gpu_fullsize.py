"""Full-size GPU parity on the four large workloads, by sampled heads.

The GPU fits, encodes and decodes the whole workload in the launch
configuration the benchmark uses.  The oracle then recomputes, for three
heads spread over the layers, everything that depends on them: the fitted
table rows (every level), every chunk's stream block, scales and int8
anchors, and the decoded fp16 tokens.  All comparisons are bit-exact.  The
long-context mixed-level workload is also decoded chunk group by chunk group
on a side stream while the next group is copied from pinned host memory,
and must equal the one-shot decode.
"""
import time

import numpy as np
import pytest

from kv_cache_compression_02_gb300 import cachegen as cg
from kv_cache_compression_02_gb300 import synth
from kv_cache_compression_02_gb300 import workloads as W
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu


def _pad16(v):
    return (v + 15) // 16 * 16


def _sample_heads(w):
    return [(0, 0, 0), (w.L // 2, 1, w.H // 2), (w.L - 1, 1, w.H - 1)]


class Run:
    """GPU fit + encode (one container per level set) + decode of a workload."""

    def __init__(self, w):
        T = gu.torch()
        gu.ready()
        self.w = w
        self.host = T.empty(w.elements, dtype=T.int16, pin_memory=True)
        synth.fill(w.gen, self.host.data_ptr())
        self.kv = self.host.cuda()
        self.cfg = cg.Config.from_workload(w)
        self.tables = cg.empty_u8(cg.cg_tables_bytes(self.cfg))
        ws = cg.empty_u8(cg.cg_workspace_bytes(self.cfg, cg.CG_OP_FIT))
        cg.check(cg.cg_fit_tables(self.cfg, self.kv, self.tables, ws), "fit")
        T.cuda.synchronize()
        assert cg.cg_read_status(ws) == cg.CG_OK
        del ws
        self.tables_host = self.tables.cpu().numpy()

    def encode(self, levels):
        T = gu.torch()
        out = cg.empty_u8(cg.cg_encode_bound(self.cfg))
        nb = T.zeros(1, dtype=T.int64, device="cuda")
        ws = cg.empty_u8(cg.cg_workspace_bytes(self.cfg, cg.CG_OP_ENCODE))
        cg.check(cg.cg_encode(self.cfg, self.tables, self.kv, levels, out, nb, ws), "encode")
        T.cuda.synchronize()
        assert cg.cg_read_status(ws) == cg.CG_OK
        del ws
        n = int(nb.item())
        return out[:n]

    def decode(self, cont_dev, k0=0, k1=-1, out=None):
        T = gu.torch()
        out = T.empty_like(self.kv) if out is None else out
        ws = cg.empty_u8(cg.cg_workspace_bytes(self.cfg, cg.CG_OP_DECODE))
        cg.check(cg.cg_decode(self.cfg, self.tables, cont_dev, cont_dev.numel(), k0, k1, out, ws), "decode")
        T.cuda.synchronize()
        assert cg.cg_read_status(ws) == cg.CG_OK
        return out


def _check_heads(orc, run, cont_host, levels, decoded_dev):
    w = run.w
    cd = orc.Codec(w.L, w.H, w.d, w.S, w.C, w.G, w.R)
    step_, recip, cdf = orc.tables_views(run.tables_host, cd, w.n_levels)
    lm = w.layer_mult_array()
    hostkv = run.host.numpy().view(np.uint16)
    nstr = w.L * 2 * w.H
    chunk_off = cont_host[64:64 + 8 * w.n_chunks].view(np.uint64)
    for (l, kv, h) in _sample_heads(w):
        si = (l * 2 + kv) * w.H + h
        head = hostkv[si * w.S * w.d:(si + 1) * w.S * w.d].reshape(w.S, w.d)
        mult = lm[l, kv] if lm is not None else [0.5, 1.0, 2.0][(3 * l) // w.L]
        c0 = h * w.d
        for lv in range(w.n_levels):
            rc, st, rp, cf = orc.fit_head(cd, w.level_base[lv], mult, head)
            assert rc == 0
            assert np.array_equal(st, step_[lv, l, kv, c0:c0 + w.d]), (l, kv, h, lv)
            assert np.array_equal(rp, recip[lv, l, kv, c0:c0 + w.d])
            assert np.array_equal(cf, cdf[lv, l, kv, c0:c0 + w.d])
        dec_head = decoded_dev[si * w.S * w.d:(si + 1) * w.S * w.d].cpu().numpy().view(np.uint16).reshape(w.S, w.d)
        ref_head = np.zeros((w.S, w.d), np.uint16)
        for k in range(w.n_chunks):
            lv = int(levels[k])
            ntok = min(w.C, w.S - k * w.C)
            ng = -(-ntok // w.G)
            base = int(chunk_off[k])
            sec_anc = 16 + _pad16(4 * nstr * w.d)
            sec_off = sec_anc + _pad16(nstr * ng * w.d)
            so = int(cont_host[base + sec_off + 4 * si: base + sec_off + 4 * si + 4].view(np.uint32)[0])
            n, blk, s, anc = orc.encode_stream(cd, head, k, step_[lv, l, kv, c0:c0 + w.d],
                                               recip[lv, l, kv, c0:c0 + w.d], cdf[lv, l, kv, c0:c0 + w.d])
            assert n > 0
            assert np.array_equal(cont_host[base + so: base + so + n], blk), (l, kv, h, k)
            gs = cont_host[base + 16 + 4 * si * w.d: base + 16 + 4 * (si + 1) * w.d].view(np.float32)
            assert np.array_equal(gs, s)
            ga = cont_host[base + sec_anc + si * ng * w.d: base + sec_anc + (si + 1) * ng * w.d].view(np.int8)
            assert np.array_equal(ga.reshape(ng, w.d), anc)
            rc = orc.decode_stream(cd, cont_host[base + so: base + so + n], k, step_[lv, l, kv, c0:c0 + w.d],
                                   cdf[lv, l, kv, c0:c0 + w.d], gs, ga.reshape(ng, w.d), ref_head)
            assert rc == 0
        assert np.array_equal(dec_head, ref_head), (l, kv, h)


@pytest.mark.parametrize("w", [W.LLAMA7B, W.LLAMA3_70B], ids=lambda w: w.name)
def test_fullsize_single_level(orc, w):
    run = Run(w)
    levels = w.levels_for()
    cont = run.encode(levels)
    decoded = run.decode(cont)
    cont_host = cont.cpu().numpy()
    assert w.fp16_bytes / cont_host.size > 2.5
    _check_heads(orc, run, cont_host, levels, decoded)


def test_fullsize_three_levels(orc):
    """Llama-3-8B shape: each chunk encoded at all three levels, each
    level's container decoded and checked on its own."""
    w = W.LLAMA3_8B
    run = Run(w)
    sizes = []
    for lv in range(w.n_levels):
        levels = w.levels_for(lv)
        cont = run.encode(levels)
        decoded = run.decode(cont)
        cont_host = cont.cpu().numpy()
        sizes.append(cont_host.size)
        _check_heads(orc, run, cont_host, levels, decoded)
        del decoded, cont
    assert sizes[0] > sizes[1] > sizes[2]  # coarser steps, smaller streams


def test_fullsize_mixed_levels_streamed(orc):
    """Long context, one of four levels per chunk; decoded in chunk groups on
    a side stream overlapped with the next group's host-to-device copy."""
    T = gu.torch()
    w = W.LONGCTX_MIXED
    run = Run(w)
    levels = w.levels_for()
    cont = run.encode(levels)
    n = cont.numel()
    cont_host = T.empty(n, dtype=T.uint8, pin_memory=True)
    cont_host.copy_(cont)
    one_shot = run.decode(cont)
    ch = cont_host.numpy()
    offs = [int(v) for v in ch[64:64 + 8 * w.n_chunks].view(np.uint64)] + [n]

    dev = cg.empty_u8(n)
    out = T.zeros_like(run.kv)
    ws = cg.empty_u8(cg.cg_workspace_bytes(run.cfg, cg.CG_OP_DECODE))
    copy_s, dec_s = T.cuda.Stream(), T.cuda.Stream()
    streamed = {}
    for group, rep in ((8, 0), (8, 1), (16, 0), (16, 1), (32, 0), (32, 1)):  # the second of each is timed
        out.zero_()
        T.cuda.synchronize()
        t0 = time.perf_counter()
        for g0 in range(0, w.n_chunks, group):
            g1 = min(g0 + group, w.n_chunks)
            lo = 0 if g0 == 0 else offs[g0]
            with T.cuda.stream(copy_s):
                dev[lo:offs[g1]].copy_(cont_host[lo:offs[g1]], non_blocking=True)
                ev = T.cuda.Event()
                ev.record(copy_s)
            dec_s.wait_event(ev)
            cg.check(cg.cg_decode(run.cfg, run.tables, dev, n, g0, g1, out, ws, dec_s), "decode group")
        T.cuda.synchronize()
        if rep:
            streamed[group] = time.perf_counter() - t0
        assert cg.cg_read_status(ws) == cg.CG_OK
        assert T.equal(out, one_shot)
    # the parts alone: the container's host-to-device copy, and the one-shot
    # decode from device memory
    T.cuda.synchronize()
    t0 = time.perf_counter()
    dev.copy_(cont_host, non_blocking=True)
    T.cuda.synchronize()
    t_copy = time.perf_counter() - t0
    t0 = time.perf_counter()
    cg.check(cg.cg_decode(run.cfg, run.tables, dev, n, 0, -1, out, ws), "decode")
    T.cuda.synchronize()
    t_dec = time.perf_counter() - t0
    # one cg_decode reading the container straight from pinned host memory
    out.zero_()
    T.cuda.synchronize()
    t0 = time.perf_counter()
    cg.check(cg.cg_decode(run.cfg, run.tables, cg.cg_host_mapped(cont_host), n, 0, -1, out, ws), "host decode")
    T.cuda.synchronize()
    direct = time.perf_counter() - t0
    assert cg.cg_read_status(ws) == cg.CG_OK
    assert T.equal(out, one_shot)
    print(f"\ncontainer {n / 1e9:.2f} GB; alone: copy {t_copy * 1e3:.1f} ms, decode {t_dec * 1e3:.1f} ms; "
          f"one decode from the pinned host container: {direct * 1e3:.1f} ms "
          f"({w.fp16_bytes / direct / 1e9:.0f} GB/s of fp16)")
    for group, t in streamed.items():
        print(f"streamed decode of {w.n_chunks} chunks in groups of {group}: {t * 1e3:.1f} ms "
              f"({w.fp16_bytes / t / 1e9:.0f} GB/s of fp16); overlap efficiency max(copy, decode) / streamed "
              f"= {max(t_copy, t_dec) / t:.2f}")
    _check_heads(orc, run, ch, levels, out)
