"""Full-size parity of a GPU container with the CPU oracle, stream by stream,
on every host core -- test infrastructure (imported by the GPU tests only).

Given the GPU's tables, container and decoded KV of a workload, one spawned
oracle process per host core takes heads in turn and, for each head
(layer, K/V, head): regenerates its fp16 values from the seeded generator,
refits its table rows at every level and compares them with the GPU's,
re-encodes every chunk's stream with the GPU's table rows and compares the
stream block, scales and anchors byte for byte, and decodes the container's
own stream blocks with the oracle and compares the result with the GPU's
decoded tokens.  The parent then checks the chunk index and stream offsets
against the oracle's stream lengths, and sums the per-table symbol counts
into the entropy bound of the coded symbols: H/8 + 4 bytes per escape + the
container's structural bytes (headers, index, scales, anchors, stream
headers), the size an ideal coder of each table's empirical distribution
would reach (Guide to CacheGen, pillar 3).  Nothing here calls the CUDA
library; the GPU side is handed in as tensors.
"""
from __future__ import annotations

import multiprocessing as mp
import os
import sys
from multiprocessing import shared_memory

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

_W = {}  # a worker's attached buffers and views


def _pad16(v):
    return (v + 15) // 16 * 16


def _init(w, names, sizes, levels, slot_heads, kv_name):
    sys.path.insert(0, ROOT)
    import oracle
    cd = oracle.Codec(w.L, w.H, w.d, w.S, w.C, w.G, w.R)
    shms = {k: shared_memory.SharedMemory(name=n) for k, n in names.items()}
    if kv_name:
        shms["kv"] = shared_memory.SharedMemory(name=kv_name)
        _W["kv"] = np.ndarray((w.L * 2 * w.H, w.S, w.d), np.uint16, buffer=shms["kv"].buf)
    tables = np.ndarray(sizes["tables"], np.uint8, buffer=shms["tables"].buf)
    cont = np.ndarray(sizes["cont"], np.uint8, buffer=shms["cont"].buf)
    dec = np.ndarray((slot_heads, w.S, w.d), np.uint16, buffer=shms["dec"].buf)
    _W.update(w=w, cd=cd, shms=shms, tables=tables, cont=cont, dec=dec, levels=np.asarray(levels, np.uint8),
              views=oracle.tables_views(tables, cd, w.n_levels))


def _head(task):
    """Check head si (slot: its place in the decoded batch, or -1 to skip the
    decode); returns (si, errors, stream lengths [nk], stats fields, entropy
    bits)."""
    import oracle
    from kv_cache_compression_02_gb300 import synth
    si, slot, check_tables = task
    w, cd, cont, levels = _W["w"], _W["cd"], _W["cont"], _W["levels"]
    step_, recip, cdf = _W["views"]
    L, H, d, S = w.L, w.H, w.d, w.S
    l, kv, h = si // (2 * H), (si // H) % 2, si % H
    head = _W["kv"][si] if "kv" in _W else synth.head(w.gen, l, kv, h)
    lm = w.layer_mult_array()
    mult = lm[l, kv] if lm is not None else [0.5, 1.0, 2.0][(3 * l) // L]
    c0 = h * d
    errs = []
    if check_tables:
        for lv in range(w.n_levels):
            rc, st, rp, cf = oracle.fit_head(cd, w.level_base[lv], mult, head)
            if rc or not (np.array_equal(st, step_[lv, l, kv, c0:c0 + d]) and
                          np.array_equal(rp, recip[lv, l, kv, c0:c0 + d]) and
                          np.array_equal(cf, cdf[lv, l, kv, c0:c0 + d])):
                errs.append(f"tables of head {si} level {lv}")
    nstr = L * 2 * H
    counts = np.zeros((w.n_levels, d, 256), np.uint64)
    stats = oracle.Stats()
    ref = np.zeros((S, d), np.uint16) if slot >= 0 else None
    chunk_off = cont[64:64 + 8 * w.n_chunks].view(np.uint64)
    lens = np.zeros(w.n_chunks, np.int64)
    for k in range(w.n_chunks):
        v = int(levels[k])
        ntok = min(w.C, S - k * w.C)
        ng = -(-ntok // w.G)
        base = int(chunk_off[k])
        sec_anc = 16 + _pad16(4 * nstr * d)
        sec_off = sec_anc + _pad16(nstr * ng * d)
        so = int(cont[base + sec_off + 4 * si: base + sec_off + 4 * si + 4].view(np.uint32)[0])
        n, blk, s, anc = oracle.encode_stream(cd, head, k, step_[v, l, kv, c0:c0 + d], recip[v, l, kv, c0:c0 + d],
                                              cdf[v, l, kv, c0:c0 + d], symcount=counts[v], stats=stats)
        lens[k] = n
        if n <= 0:
            errs.append(f"oracle encode of head {si} chunk {k}: {n}")
            continue
        gblk = cont[base + so: base + so + n]
        gs = cont[base + 16 + 4 * si * d: base + 16 + 4 * (si + 1) * d].view(np.float32)
        ga = cont[base + sec_anc + si * ng * d: base + sec_anc + (si + 1) * ng * d].view(np.int8).reshape(ng, d)
        if not np.array_equal(gblk, blk):
            errs.append(f"stream of head {si} chunk {k}")
        if not np.array_equal(gs, s) or not np.array_equal(ga, anc):
            errs.append(f"scales/anchors of head {si} chunk {k}")
        if ref is not None and oracle.decode_stream(cd, gblk, k, step_[v, l, kv, c0:c0 + d], cdf[v, l, kv, c0:c0 + d],
                                                    gs, ga, ref) != 0:
            errs.append(f"oracle decode of head {si} chunk {k}")
    if ref is not None and not np.array_equal(_W["dec"][slot], ref):
        bad = np.argwhere(_W["dec"][slot] != ref)
        errs.append(f"decoded head {si}: {len(bad)} values differ, first at token/lane {tuple(bad[0])}")
    ent = sum(oracle.table_entropy(counts[v, j]) for v in range(w.n_levels) for j in range(d) if counts[v, j].any())
    st = (stats.n_symbols, stats.n_esc, stats.n_words, stats.fixed_bytes, stats.state_bytes, stats.pad_bytes)
    return si, errs, lens, st, ent


def verify(w, tables, cont, levels, decoded, tables_every=1, decode_every=1, procs=None, batch=64, kv_shm=None):
    """Compare every stream of container `cont` (uint8 tensor, GPU or host)
    with the oracle.  tables: uint8 tensor; decoded: the GPU's decoded KV
    (int16/uint16 tensor [L*2*H*S*d]); heads with si % decode_every == 0 also
    have their decoded tokens compared, and si % tables_every == 0 their
    table rows.  kv_shm: name of a shared-memory block holding the input KV
    (the heads are regenerated when it is None).  Returns a report dict
    (errors listed, not raised)."""
    import torch
    sys.path.insert(0, ROOT)
    import oracle
    procs = procs or os.cpu_count() or 1
    nstr, S, d = w.L * 2 * w.H, w.S, w.d
    sizes = {"tables": tables.numel(), "cont": cont.numel(), "dec": batch * S * d * 2}
    shms = {k: shared_memory.SharedMemory(create=True, size=max(v, 1)) for k, v in sizes.items()}
    try:
        for k, src in (("tables", tables), ("cont", cont)):
            torch.frombuffer(shms[k].buf, dtype=torch.uint8, count=src.numel()).copy_(src.reshape(-1))
        dec_host = torch.frombuffer(shms["dec"].buf, dtype=torch.int16, count=batch * S * d)
        flat = decoded.reshape(-1).view(torch.int16)
        names = {k: v.name for k, v in shms.items()}
        ctx = mp.get_context("spawn")
        errors, lens = [], np.zeros((w.n_chunks, nstr), np.int64)
        tot = np.zeros(6, np.int64)
        ent = 0.0
        with ctx.Pool(procs, initializer=_init, initargs=(w, names, sizes, list(levels), batch, kv_shm)) as pool:
            for s0 in range(0, nstr, batch):
                heads = list(range(s0, min(s0 + batch, nstr)))
                tasks = []
                for j, si in enumerate(heads):
                    slot = j if si % decode_every == 0 else -1
                    if slot >= 0:
                        dec_host[j * S * d:(j + 1) * S * d].copy_(flat[si * S * d:(si + 1) * S * d])
                    tasks.append((si, slot, si % tables_every == 0))
                for si, errs, ln, st, e in pool.map(_head, tasks, chunksize=1):
                    errors += errs
                    lens[:, si] = ln
                    tot += np.asarray(st, np.int64)
                    ent += e
        # the index: chunk offsets and each chunk's stream offsets follow from
        # the oracle's stream lengths
        c = np.ndarray(cont.numel(), np.uint8, buffer=shms["cont"].buf)
        chunk_off = c[64:64 + 8 * w.n_chunks].view(np.uint64).astype(np.int64)
        for k in range(w.n_chunks):
            ntok = min(w.C, S - k * w.C)
            ng = -(-ntok // w.G)
            sec_off = 16 + _pad16(4 * nstr * d) + _pad16(nstr * ng * d)
            fixed = sec_off + _pad16(4 * nstr)
            hdr = c[chunk_off[k]:chunk_off[k] + 16].view(np.uint32)
            if (hdr[0] & 0xFFFF) != levels[k] or hdr[1] != k * w.C or hdr[2] != ntok or hdr[3] != ng:
                errors.append(f"chunk {k} header")
            so = c[chunk_off[k] + sec_off:chunk_off[k] + sec_off + 4 * nstr].view(np.uint32).astype(np.int64)
            if not np.array_equal(so, fixed + np.concatenate([[0], np.cumsum(lens[k])[:-1]])):
                errors.append(f"chunk {k} stream offsets")
            end = chunk_off[k + 1] if k + 1 < w.n_chunks else cont.numel()
            if end != chunk_off[k] + fixed + lens[k].sum():
                errors.append(f"chunk {k} size")
        cd = oracle.Codec(w.L, w.H, w.d, w.S, w.C, w.G, w.R)
        st = oracle.Stats(ent, *[int(v) for v in tot[:3]], int(tot[3]) + oracle.container_fixed_bytes(cd),
                          *[int(v) for v in tot[4:]])
        bound = oracle.entropy_bound_bytes(st)
        return {"workload": w.name, "levels": sorted(set(int(v) for v in levels)), "streams": nstr * w.n_chunks,
                "container_bytes": int(cont.numel()), "bound_bytes": bound,
                "actual_over_bound": cont.numel() / bound,
                "actual_over_bound_incl_tables": (cont.numel() + tables.numel()) / (bound + tables.numel()),
                "escapes": int(tot[1]), "errors": errors,
                "decoded_heads": len(range(0, nstr, decode_every)), "table_heads": len(range(0, nstr, tables_every))}
    finally:
        for v in shms.values():
            v.close()
            v.unlink()
