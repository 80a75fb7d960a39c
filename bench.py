"""Throughput of the CacheGen codec on one GB300 per rank.

One step = one pass of the whole hot path over the Llama-3-70B-shaped KV
(L=80, H_kv=8, d=128, S=32768, fp16, 10.7 GB): cg_fit_tables (channel
statistics, anchor scales, histograms, 16-bit CDFs), cg_encode (anchors,
closed-loop deltas, rANS streams, size scan, compaction) and cg_decode
(rANS decode + fused dequantisation into the KV layout).  Inputs are
resident in HBM when the timed region starts and are larger than L2.

The headline value is decode throughput (fp16 GB/s written by cg_decode);
encode and fit throughput, the compression ratio (with and without the
tables), roofline fractions, an end-to-end figure through host
buffers, the same decode in layer groups (time to the first group) and into
a paged (block-table) cache, and a bandwidth-adaptive streaming run (chunk
levels chosen by the host controller over a simulated link, the planned
container encoded and decoded on the GPU) are reported beside it.  (The
container's size against the entropy bound of its coded symbols is a gate of
the oracle tests, which reproduce the bytes exactly.)  `--impl reference`
times the CPU oracle on every host core, on a bounded sample of the same
workload, instead.

Multi-GPU: every rank codes its own copy of the workload (independent
problems, no collective on the data path); value = all ranks' bytes / the
slowest rank's time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "decode & encode GB/s of fp16 KV (70B shape, 1 GB300); ratio; % HBM roofline"


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="llama3_70b_L80_H8_d128_S32768")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--e2e-steps", type=int, default=3)
    ap.add_argument("--no-paged", action="store_true",
                    help="skip the layer-group, paged-cache and adaptive-streaming legs")
    ap.add_argument("--layers", type=int, default=0,
                    help="run the same workload with fewer layers (a smaller case for profiling)")
    ap.add_argument("--stream-groups", type=int, default=0,
                    help="also decode the container group by group of this many chunks on a side stream, "
                         "each group as soon as its bytes have been copied from pinned host memory")
    return ap.parse_args()


def dist_env():
    return int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)), int(os.environ.get("LOCAL_RANK", 0))


def rank_max(values, world: int, device):
    """Each value's maximum over the ranks (one all-reduce; as given at N=1):
    the job's time is its slowest rank's."""
    values = [float(v) for v in values]
    if world == 1:
        return values
    import torch
    import torch.distributed as dist
    t = torch.tensor(values, dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.tolist()


def job_gbs(bytes_per_rank: float, world: int, max_ms: float) -> float:
    """Whole-job throughput: every rank's bytes over the slowest rank's time."""
    return world * bytes_per_rank / (max_ms * 1e-3) / 1e9


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as fh:
            p = json.load(fh)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


class Clocks:
    """nvidia-smi sampling during the timed region."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, dev: int):
        self.dev = dev
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.dev), f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        self.proc.wait()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        os.unlink(self.path)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def traffic_for(kernel: str, per_launch_units: float):
    """DRAM bytes per launch from a committed ncu summary, if it was taken on
    the current kernel source (null otherwise)."""
    try:
        with open(os.path.join(ROOT, "profiles", "traffic.json")) as fh:
            t = json.load(fh)[kernel]
        src = open(os.path.join(ROOT, "kv_cache_compression_02_gb300", "csrc", t["source"]), "rb").read()
        if hashlib.sha256(src).hexdigest()[:16] != t["source_sha"]:
            return None
        return t["dram_bytes_per_unit"] * per_launch_units
    except Exception:
        return None


def generate_pinned(w, torch):
    from kv_cache_compression_02_gb300 import synth
    host = torch.empty(w.elements, dtype=torch.int16, pin_memory=True)
    t0 = time.time()
    synth.fill(w.gen, host.data_ptr())
    return host, time.time() - t0


def cpu_oracle_decode_rate(w, host_np, budget_s=10.0):
    """Single-threaded oracle decode rate (fp16 bytes/s) on a bounded sample:
    the chunk streams of successive heads, each fitted by the oracle first
    (untimed) and encoded (timed apart: the oracle's encode rate), until
    budget_s of decode time has been spent.  Returns (decode rate, decode
    seconds, streams, encode rate)."""
    import oracle
    oracle.build()
    cd = oracle.Codec(w.L, w.H, w.d, w.S, w.C, w.G, w.R)
    L, H, S, d = w.L, w.H, w.S, w.d
    spent, spent_enc, nbytes, streams = 0.0, 0.0, 0, 0
    heads = L * 2 * H
    step_ = max(1, heads // 128)
    out = np.zeros((S, d), np.uint16)
    lm = w.layer_mult_array()
    for si in range(0, heads, step_):
        l, kvi = si // (2 * H), (si // H) % 2
        head = host_np[si * S * d:(si + 1) * S * d].reshape(S, d)
        m = lm[l, kvi] if lm is not None else [0.5, 1.0, 2.0][(3 * l) // L]
        rc, st, rp, cdf = oracle.fit_head(cd, w.level_base[0], m, head)
        for k in range(cd.n_chunks):
            t0 = time.perf_counter()
            n, blk, s, anc = oracle.encode_stream(cd, head, k, st, rp, cdf)
            t1 = time.perf_counter()
            rc = oracle.decode_stream(cd, blk, k, st, cdf, s, anc, out)
            spent += time.perf_counter() - t1
            spent_enc += t1 - t0
            assert rc == 0
            nbytes += min(w.C, S - k * w.C) * d * 2
            streams += 1
            if spent >= budget_s:
                return nbytes / spent, spent, streams, nbytes / spent_enc
    return nbytes / spent, spent, streams, nbytes / spent_enc


def _oracle_worker(args):
    """One process of the all-core oracle run: heads si = first, first +
    stride, ... of workload `name`, generated here; the oracle fits and
    encodes each (untimed) and decodes its chunk streams until budget_s of
    decode time is spent.  Returns (fp16 bytes decoded, decode seconds)."""
    name, first, stride, budget_s = args
    sys.path.insert(0, ROOT)
    import oracle
    from kv_cache_compression_02_gb300 import synth, workloads as W
    w = W.BY_NAME[name]
    cd = oracle.Codec(w.L, w.H, w.d, w.S, w.C, w.G, w.R)
    out = np.zeros((w.S, w.d), np.uint16)
    spent, nbytes = 0.0, 0
    for si in range(first, w.L * 2 * w.H, stride):
        l, kv, h = si // (2 * w.H), (si // w.H) % 2, si % w.H
        head = synth.head(w.gen, l, kv, h)
        lm = w.layer_mult_array()
        m = lm[l, kv] if lm is not None else [0.5, 1.0, 2.0][(3 * l) // w.L]
        rc, st, rp, cdf = oracle.fit_head(cd, w.level_base[0], m, head)
        for k in range(cd.n_chunks):
            n, blk, sc, anc = oracle.encode_stream(cd, head, k, st, rp, cdf)
            t0 = time.perf_counter()
            assert oracle.decode_stream(cd, blk, k, st, cdf, sc, anc, out) == 0
            spent += time.perf_counter() - t0
            nbytes += min(w.C, w.S - k * w.C) * w.d * 2
            if spent >= budget_s:
                return nbytes, spent
    return nbytes, spent


def cpu_oracle_decode_rate_all_cores(name, budget_s=10.0):
    """The oracle decode on every host core at once (one spawned process per
    core, each on its own heads): summed fp16 bytes/s, and the core count."""
    import multiprocessing as mp
    import oracle
    oracle.build()
    n = os.cpu_count() or 1
    with mp.get_context("spawn").Pool(n) as pool:
        res = pool.map(_oracle_worker, [(name, i * 7, n * 7, budget_s) for i in range(n)])
    return sum(b / t for b, t in res if t > 0), n


def workload_config(w, world):
    """The bench line's config for workload w (both arms)."""
    return {"workload": w.name, "L": w.L, "H_kv": w.H, "d": w.d, "S": w.S, "C": w.C, "G": w.G,
            "levels": list(w.level_base), "chunk_levels": w.chunk_levels, "fp16_bytes": w.fp16_bytes,
            "l2": (f"inputs larger than L2 ({w.fp16_bytes / 1e9:.1f} GB)" if 2 * w.fp16_bytes >= (256 << 20)
                   else "a 256 MB buffer written between steps (inputs smaller than L2)"),
            "parallelism": f"independent replica per GPU x{world}"}


_REF = None  # a reference-arm worker's prepared streams


def _ref_init(name, nworkers, per_worker, ids):
    """Reference-arm worker: take an index from ids, then generate, fit and
    encode (untimed) the chunk-0 streams of its heads, spread over the
    layers."""
    global _REF
    sys.path.insert(0, ROOT)
    import oracle
    from kv_cache_compression_02_gb300 import synth, workloads as W
    w = W.BY_NAME[name]
    widx = ids.get()
    nsi = w.L * 2 * w.H
    stride = max(1, nsi // (nworkers * per_worker))
    cd = oracle.Codec(w.L, w.H, w.d, w.S, w.C, w.G, w.R)
    prepared = []
    for j in range(per_worker):
        si = ((widx % nworkers) + j * nworkers) * stride % nsi
        l, kv, h = si // (2 * w.H), (si // w.H) % 2, si % w.H
        head = synth.head(w.gen, l, kv, h)
        lm = w.layer_mult_array()
        m = lm[l, kv] if lm is not None else [0.5, 1.0, 2.0][(3 * l) // w.L]
        rc, st, rp, cdf = oracle.fit_head(cd, w.level_base[0], m, head)
        n, blk, sc, anc = oracle.encode_stream(cd, head, 0, st, rp, cdf)
        prepared.append((blk, st, cdf, sc, anc))
    _REF = (cd, np.zeros((w.S, w.d), np.uint16), prepared)


def _ref_step(_):
    """Decode the worker's prepared streams once; returns the fp16 bytes."""
    import oracle
    cd, out, prepared = _REF
    for blk, st, cdf, sc, anc in prepared:
        assert oracle.decode_stream(cd, blk, 0, st, cdf, sc, anc, out) == 0
    return len(prepared) * min(cd.C, cd.S) * cd.d * 2


def run_reference(args):
    """The CPU oracle on the machine's host cores (reference arm): one spawned
    process per core, each decoding the chunk-0 streams of its own heads per
    step; a step is one decode of every process's streams, timed on the
    wall clock."""
    import multiprocessing as mp
    rank, world, _ = dist_env()
    if rank != 0:
        return
    from kv_cache_compression_02_gb300 import workloads as W
    import oracle
    w = W.BY_NAME[args.workload]
    oracle.build()
    n = os.cpu_count() or 1
    per_worker = 8
    ctx = mp.get_context("spawn")
    ids = ctx.Queue()
    for i in range(n):
        ids.put(i)
    with ctx.Pool(n, initializer=_ref_init, initargs=(w.name, n, per_worker, ids)) as pool:
        for _ in range(args.warmup):
            pool.map(_ref_step, range(n), chunksize=1)
        nbytes = 0
        t0 = time.perf_counter()
        for _ in range(args.steps):
            nbytes += sum(pool.map(_ref_step, range(n), chunksize=1))
        dt = (time.perf_counter() - t0) / max(args.steps, 1)
    nbytes_step = nbytes / max(args.steps, 1)
    v = nbytes_step / dt / 1e9
    sample = (f"oracle decode of the chunk-0 streams ({w.C} tokens x {w.d} lanes) of {n * per_worker} heads "
              f"spread over the layers, {per_worker} per process, one process per core, per step")
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": v, "unit": "GB/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "u32+f32", "data": "synthetic",
        "config": dict(workload_config(w, args.gpus), sample=sample),
        "cpu_baseline": {"value": v, "unit": "GB/s", "cores": n, "kind": "oracle", "sample": sample},
        "e2e": {"value": v, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


def main():
    args = parse()
    if args.impl == "reference":
        return run_reference(args)
    import torch
    import torch.distributed as dist

    from kv_cache_compression_02_gb300 import build as cgbuild, cachegen as cg, workloads as W

    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    cgbuild.build()
    w = W.BY_NAME[args.workload]
    if args.layers:
        w = W.scaled(w, L=args.layers, name=f"{w.name}_L{args.layers}")
    dev = torch.device("cuda", local)
    stream = torch.cuda.current_stream()

    host, gen_s = generate_pinned(w, torch)
    kv = host.to(dev, non_blocking=True)
    cfg = cg.Config.from_workload(w)
    tables = cg.empty_u8(cg.cg_tables_bytes(cfg))
    ws_fit = cg.empty_u8(cg.cg_workspace_bytes(cfg, cg.CG_OP_FIT))
    ws_enc = cg.empty_u8(cg.cg_workspace_bytes(cfg, cg.CG_OP_ENCODE))
    ws_dec = cg.empty_u8(cg.cg_workspace_bytes(cfg, cg.CG_OP_DECODE))
    # the containers a step encodes and decodes: one, or (for a workload
    # coded once per level) one per level
    level_sets = ([w.levels_for(v) for v in range(w.n_levels)] if w.chunk_levels == "each"
                  else [w.levels_for()])
    nsets = len(level_sets)
    outs = [cg.empty_u8(cg.cg_encode_bound(cfg)) for _ in level_sets]
    out = outs[0]
    nbytes_d = torch.zeros(1, dtype=torch.int64, device=dev)
    kv_out = torch.empty_like(kv)
    levels = level_sets[0]
    # inputs smaller than L2: a buffer larger than L2 is written between steps
    l2_flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev) if 2 * w.fp16_bytes < (256 << 20) else None
    torch.cuda.synchronize()

    ev = {"fit": [], "enc": [[] for _ in level_sets], "dec": [[] for _ in level_sets]}
    nbytes_list = [None] * nsets

    def step(record: bool):
        e = [torch.cuda.Event(enable_timing=True) for _ in range(2 + 2 * nsets)]
        e[0].record(stream)
        cg.check(cg.cg_fit_tables(cfg, kv, tables, ws_fit, stream), "cg_fit_tables")
        e[1].record(stream)
        for j, lv_set in enumerate(level_sets):
            cg.check(cg.cg_encode(cfg, tables, kv, lv_set, outs[j], nbytes_d, ws_enc, stream), "cg_encode")
            e[2 + 2 * j].record(stream)
            if nbytes_list[j] is None:
                torch.cuda.synchronize()
                nbytes_list[j] = int(nbytes_d.item())
            cg.check(cg.cg_decode(cfg, tables, outs[j], nbytes_list[j], 0, -1, kv_out, ws_dec, stream), "cg_decode")
            e[3 + 2 * j].record(stream)
        if record:
            ev["fit"].append((e[0], e[1]))
            for j in range(nsets):
                ev["enc"][j].append((e[1 + 2 * j], e[2 + 2 * j]))
                ev["dec"][j].append((e[2 + 2 * j], e[3 + 2 * j]))
        if l2_flush is not None:
            l2_flush.zero_()

    for _ in range(max(args.warmup, 1)):
        step(False)
    torch.cuda.synchronize()
    nbytes = nbytes_list[0]
    for ws, what in ((ws_fit, "fit"), (ws_enc, "encode"), (ws_dec, "decode")):
        cg.check(cg.cg_read_status(ws), what)
    # sanity: the decode reproduces the input within the quantization error
    xs = kv[: 1 << 20].view(torch.float16).float()
    ys = kv_out[: 1 << 20].view(torch.float16).float()
    if not torch.isfinite(ys).all() or (xs - ys).abs().max().item() > 0.5 * xs.abs().max().item():
        raise RuntimeError("decoded KV does not match the input")
    # the entropy bound of each single-level container, from the fit's histograms
    ebounds = [cg.cg_entropy_bound(cfg, ws_fit, int(s_[0])) if len(set(s_.tolist())) == 1 else None
               for s_ in level_sets]

    clocks = Clocks(local)
    clocks.start()
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    t_start.record(stream)
    for _ in range(args.steps):
        step(True)
    t_end.record(stream)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    clk = clocks.stop()
    mean_ms = lambda v: sum(a.elapsed_time(b) for a, b in v) / len(v)  # noqa: E731
    ms_enc_sets = [mean_ms(v) for v in ev["enc"]]
    ms_dec_sets = [mean_ms(v) for v in ev["dec"]]
    ms = {"fit": mean_ms(ev["fit"]), "enc": sum(ms_enc_sets), "dec": sum(ms_dec_sets)}
    # the steps' own time (the L2 flush between steps, when there is one, excluded)
    ms_step = (t_start.elapsed_time(t_end) / args.steps if l2_flush is None
               else ms["fit"] + ms["enc"] + ms["dec"])
    for ws, what in ((ws_fit, "fit"), (ws_enc, "encode"), (ws_dec, "decode")):
        cg.check(cg.cg_read_status(ws), what)

    # end to end through host buffers.  Headline: one cg_decode whose
    # container and output both sit in pinned host memory, mapped into the
    # device's address space: the decoder reads the container's words and
    # writes the fp16 tokens across the host link itself, with no staging
    # copy.  Beside it: the pipelined form (per 4-chunk group, the container
    # bytes go to the device on one stream, the group decodes on another and
    # its tokens come back on a third as one strided copy) and the serial
    # sequence (container H2D, one cg_decode, KV D2H).
    import ctypes
    import glob
    cont_host = torch.empty(nbytes, dtype=torch.uint8, pin_memory=True)
    cont_host.copy_(out[:nbytes])
    out_host = torch.empty(kv.numel(), dtype=torch.int16, pin_memory=True)
    cont_dev = cg.empty_u8(nbytes)
    offs = [int(v) for v in cont_host[64:64 + 8 * w.n_chunks].numpy().view(np.uint64)] + [nbytes]
    cudart = ctypes.CDLL(sorted(glob.glob(os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"),
                                                       "lib64", "libcudart.so.*")))[-1])
    cudart.cudaMemcpy2DAsync.restype = ctypes.c_int
    cudart.cudaMemcpy2DAsync.argtypes = [ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p, ctypes.c_size_t,
                                         ctypes.c_size_t, ctypes.c_size_t, ctypes.c_int, ctypes.c_void_p]
    cont_map, out_map = cg.cg_host_mapped(cont_host), cg.cg_host_mapped(out_host)  # for the direct decode
    e2e_groups = [(k0, min(k0 + 4, w.n_chunks)) for k0 in range(0, w.n_chunks, 4)]
    h2d_s, d2h_s = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    row_bytes = w.S * w.d * 2
    torch.cuda.synchronize()

    def e2e_pipelined():
        h2d_s.wait_stream(stream)  # the copies start inside the timed region
        for k0, k1 in e2e_groups:
            lo_b = 0 if k0 == 0 else offs[k0]  # the first group carries the header and chunk index
            with torch.cuda.stream(h2d_s):
                cont_dev[lo_b:offs[k1]].copy_(cont_host[lo_b:offs[k1]], non_blocking=True)
            arrived = torch.cuda.Event()
            arrived.record(h2d_s)
            stream.wait_event(arrived)
            cg.check(cg.cg_decode(cfg, tables, cont_dev, nbytes, k0, k1, kv_out, ws_dec, stream), "cg_decode")
            decoded = torch.cuda.Event()
            decoded.record(stream)
            d2h_s.wait_event(decoded)
            t0_, t1_ = k0 * w.C, min(k1 * w.C, w.S)
            off = t0_ * w.d * 2
            rc = cudart.cudaMemcpy2DAsync(out_host.data_ptr() + off, row_bytes, kv_out.data_ptr() + off, row_bytes,
                                          (t1_ - t0_) * w.d * 2, w.L * 2 * w.H, 2, ctypes.c_void_p(d2h_s.cuda_stream))
            if rc != 0:
                raise RuntimeError(f"cudaMemcpy2DAsync failed ({rc})")
        stream.wait_stream(d2h_s)

    def e2e_serial():
        cont_dev.copy_(cont_host, non_blocking=True)
        cg.check(cg.cg_decode(cfg, tables, cont_dev, nbytes, 0, -1, kv_out, ws_dec, stream), "cg_decode")
        out_host.copy_(kv_out, non_blocking=True)

    def e2e_direct():
        cg.check(cg.cg_decode(cfg, tables, cont_map, nbytes, 0, -1, out_map, ws_dec, stream), "cg_decode")

    e2e_ms, e2e_pipe_ms, e2e_serial_ms = [], [], []
    for fn, acc in ((e2e_pipelined, e2e_pipe_ms), (e2e_serial, e2e_serial_ms), (e2e_direct, e2e_ms)):
        if fn is e2e_direct:
            out_host.zero_()  # the check below then sees only what the direct decode wrote
        for i in range(args.e2e_steps + 1):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            fn()
            b.record(stream)
            torch.cuda.synchronize()
            if i:
                acc.append(a.elapsed_time(b))
        cg.check(cg.cg_read_status(ws_dec), "decode (e2e)")
    for lo_ in (0, kv.numel() // 2, kv.numel() - (1 << 24)):  # spot check three 32 MB windows
        if not torch.equal(out_host[lo_:lo_ + (1 << 24)], kv_out[lo_:lo_ + (1 << 24)].cpu()):
            raise RuntimeError("end-to-end copy differs from the decoded KV")
    cg.check(cg.cg_read_status(ws_dec), "decode (e2e)")
    # the host link alone, by the copy engines, on the same buffers: the
    # bound the end-to-end decode is measured against
    link = {}
    for name, fn, nb_ in (("h2d_gbs", lambda: cont_dev.copy_(cont_host, non_blocking=True), nbytes),
                          ("d2h_gbs", lambda: out_host.copy_(kv_out, non_blocking=True), kv.numel() * 2)):
        ts = []
        for i in range(3):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            with torch.cuda.stream(stream):
                fn()
            b.record(stream)
            torch.cuda.synchronize()
            if i:
                ts.append(a.elapsed_time(b))
        link[name] = nb_ / (statistics.mean(ts) * 1e-3) / 1e9

    # chunk-group streaming: group g's container bytes are copied from pinned
    # host memory on one stream, and the group decodes as soon as they have
    # landed, while group g + 1 is being copied; the groups' decodes alternate
    # between two streams, each with its own workspace, so that a group's
    # launches can fill the SMs the previous group's last wave leaves idle
    # (the groups write disjoint tokens); against the copy alone and the
    # one-shot decode from device memory
    streamed = None
    if args.stream_groups:
        G = args.stream_groups
        copy_s, dec_s = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
        dec_s2 = torch.cuda.Stream(device=dev)
        ws_dec2 = cg.empty_u8(cg.cg_workspace_bytes(cfg, cg.CG_OP_DECODE))
        win = [(lo_, lo_ + (1 << 22)) for lo_ in (0, kv.numel() // 2, kv.numel() - (1 << 22))]
        ref = [kv_out[a_:b_].clone() for a_, b_ in win]  # kv_out holds the serial end-to-end decode

        def timed(fn, s0, s1):
            torch.cuda.synchronize()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(s0)
            fn()
            b.record(s1)
            torch.cuda.synchronize()
            return a.elapsed_time(b)

        def stream_groups():
            for gi, g0 in enumerate(range(0, w.n_chunks, G)):
                g1 = min(g0 + G, w.n_chunks)
                lo_b = 0 if g0 == 0 else offs[g0]  # the first group carries the header and chunk index
                with torch.cuda.stream(copy_s):
                    cont_dev[lo_b:offs[g1]].copy_(cont_host[lo_b:offs[g1]], non_blocking=True)
                arrived = torch.cuda.Event()
                arrived.record(copy_s)
                ds, wsd = (dec_s, ws_dec) if gi % 2 == 0 else (dec_s2, ws_dec2)
                ds.wait_event(arrived)
                cg.check(cg.cg_decode(cfg, tables, cont_dev, nbytes, g0, g1, kv_out, wsd, ds), "cg_decode")
            done2 = torch.cuda.Event()
            done2.record(dec_s2)
            dec_s.wait_event(done2)  # the end event, on dec_s, follows both decode streams

        def copy_alone():
            with torch.cuda.stream(copy_s):
                cont_dev.copy_(cont_host, non_blocking=True)

        def decode_alone():
            cg.check(cg.cg_decode(cfg, tables, cont_dev, nbytes, 0, -1, kv_out, ws_dec, dec_s), "cg_decode")

        kv_out.zero_()
        t_stream = [timed(stream_groups, copy_s, dec_s) for _ in range(3)]
        cg.check(cg.cg_read_status(ws_dec), "decode (streamed)")
        cg.check(cg.cg_read_status(ws_dec2), "decode (streamed)")
        for (a_, b_), r_ in zip(win, ref):
            if not torch.equal(kv_out[a_:b_], r_):
                raise RuntimeError("streamed decode differs from the one-shot decode")
        t_copy = min(timed(copy_alone, copy_s, copy_s) for _ in range(3))
        t_dec = min(timed(decode_alone, dec_s, dec_s) for _ in range(3))
        t_s = min(t_stream)
        streamed = {"groups_of_chunks": G, "ms": t_s, "copy_ms": t_copy, "decode_ms": t_dec,
                    "overlap_efficiency": max(t_copy, t_dec) / t_s, "fp16_gbs": w.fp16_bytes / (t_s * 1e-3) / 1e9,
                    "what": "container copied group by group from pinned host memory on one stream, each group "
                            "decoded once its bytes have landed, on two streams in turn (a workspace each); "
                            "efficiency = max(copy alone, one-shot decode) / streamed"}
        del ref

    # the same decode in layer groups, in execution order: 19 layers (304
    # CTAs, two full waves) per launch, an event after each group
    lgroups = None
    if not args.no_paged:
        per = 19
        bounds = [(l0, min(l0 + per, w.L)) for l0 in range(0, w.L, per)]
        lev = []
        for i in range(max(args.warmup, 1) + args.steps):
            evs = [torch.cuda.Event(enable_timing=True) for _ in range(len(bounds) + 1)]
            evs[0].record(stream)
            for gi, (l0, l1) in enumerate(bounds):
                cg.check(cg.cg_decode_layers(cfg, tables, out, nbytes, 0, -1, l0, l1, kv_out, ws_dec, stream),
                         "cg_decode_layers")
                evs[gi + 1].record(stream)
            if i >= max(args.warmup, 1):
                lev.append(evs)
        torch.cuda.synchronize()
        cg.check(cg.cg_read_status(ws_dec), "decode (layer groups)")
        first = statistics.mean(e[0].elapsed_time(e[1]) for e in lev)
        total = statistics.mean(e[0].elapsed_time(e[-1]) for e in lev)
        lgroups = {"layers_per_group": per, "groups": len(bounds), "first_group_ms": first, "all_groups_ms": total,
                   "fp16_gbs": w.fp16_bytes / (total * 1e-3) / 1e9}

    # the same decode into a paged cache: 16-token blocks, shuffled block table
    paged = None
    if not args.no_paged:
        bt = 16
        n_lblk = -(-w.S // bt)
        pools = torch.empty((w.L * 2, n_lblk, w.H, bt, w.d), dtype=torch.int16, device=dev)
        ptrs = torch.tensor([pools.data_ptr() + i * pools.stride(0) * 2 for i in range(w.L * 2)],
                            dtype=torch.int64, device=dev)
        table = torch.randperm(n_lblk, generator=torch.Generator().manual_seed(0)).to(torch.int32).to(dev)
        pev = []
        for i in range(max(args.warmup, 1) + args.steps):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            cg.check(cg.cg_decode_paged(cfg, tables, out, nbytes, 0, -1, ptrs, table, bt, n_lblk, ws_dec, stream),
                     "cg_decode_paged")
            b.record(stream)
            if i >= max(args.warmup, 1):
                pev.append((a, b))
        torch.cuda.synchronize()
        cg.check(cg.cg_read_status(ws_dec), "decode (paged)")
        # spot check: a few logical blocks hold the contiguous decode's rows
        kvo = kv_out.view(w.L * 2, w.H, w.S, w.d)
        for lb in (0, n_lblk // 2, n_lblk - 1):
            t0, t1 = lb * bt, min(w.S, lb * bt + bt)
            if not torch.equal(pools[:, int(table[lb]), :, : t1 - t0], kvo[:, :, t0:t1]):
                raise RuntimeError("paged decode differs from the contiguous decode")
        ms_paged = statistics.mean(a.elapsed_time(b) for a, b in pev)
        paged = {"ms": ms_paged, "fp16_gbs": w.fp16_bytes / (ms_paged * 1e-3) / 1e9, "block_tokens": bt,
                 "table": "random permutation of the sequence's blocks"}
        del pools

    # bandwidth-adaptive levels over a simulated link: chunk sizes from GPU
    # encodes at four levels, the host controller picks a level per chunk,
    # the planned mixed-level container is GPU-encoded and decoded
    adaptive = None
    if not args.no_paged:
        lb4 = (0.05, 0.1, 0.2, 0.4)
        cfg4 = cg.Config.from_workload(w, level_base=lb4)
        tb4 = cg.empty_u8(cg.cg_tables_bytes(cfg4))
        ws4 = cg.empty_u8(max(cg.cg_workspace_bytes(cfg4, op) for op in (cg.CG_OP_FIT, cg.CG_OP_ENCODE,
                                                                          cg.CG_OP_DECODE)))
        cg.check(cg.cg_fit_tables(cfg4, kv, tb4, ws4, stream), "cg_fit_tables (4 levels)")
        nk = w.n_chunks
        sizes = np.zeros((nk, len(lb4)), np.int64)
        singles = []  # the context encoded once per level
        for lv in range(len(lb4)):
            cg.check(cg.cg_encode(cfg4, tb4, kv, np.full(nk, lv, np.uint8), out, nbytes_d, ws4, stream),
                     "cg_encode (one level)")
            torch.cuda.synchronize()
            cg.check(cg.cg_read_status(ws4), "encode (one level)")
            n_lv = int(nbytes_d.item())
            singles.append(out[:n_lv].clone())
            offs = np.append(out[64:64 + 8 * nk].cpu().numpy().view(np.uint64).astype(np.int64), n_lv)
            sizes[:, lv] = np.diff(offs)
            sizes[0, lv] += offs[0]  # the header and chunk index go out with chunk 0
        nominal, low = 50e9, 12.5e9  # 400 Gb/s, dropping to 100 Gb/s for 25 ms after 20 ms
        trace = [(0.020, nominal), (0.025, low), (1.0, nominal)]
        dec = [ms["dec"] * 1e-3 / nk] * nk  # the measured decode, spread evenly over the chunks
        deadline = 1.1 * sizes[:, 1].sum() / nominal + dec[-1]
        rc, lv_plan, _, total = cg.cg_plan_levels(sizes, trace, nominal, deadline, dec)
        cg.check(rc, "cg_plan_levels")
        fixed = {f"level_{lv}": cg.cg_simulate_stream(sizes, trace, [lv] * nk, dec)[2] for lv in range(len(lb4))}
        # the planned container from the per-level ones (device copies), checked
        # against a direct encode with the planned levels
        ws_a = cg.empty_u8(cg.cg_workspace_bytes(cfg4, cg.CG_OP_ASSEMBLE))
        asm = cg.empty_u8(cg.cg_encode_bound(cfg4))
        nb_a = torch.zeros(1, dtype=torch.int64, device=dev)
        ta, tb_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        ta.record(stream)
        cg.check(cg.cg_assemble(cfg4, singles, lv_plan, asm, nb_a, ws_a, stream), "cg_assemble")
        tb_.record(stream)
        cg.check(cg.cg_encode(cfg4, tb4, kv, lv_plan, out, nbytes_d, ws4, stream), "cg_encode (planned)")
        torch.cuda.synchronize()
        cg.check(cg.cg_read_status(ws_a), "assemble (planned)")
        n_plan = int(nbytes_d.item())
        if int(nb_a.item()) != n_plan or not torch.equal(asm[:n_plan], out[:n_plan]):
            raise RuntimeError("assembled container differs from the direct encode")
        assemble_ms = ta.elapsed_time(tb_)
        del asm, singles
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        cg.check(cg.cg_decode(cfg4, tb4, out, n_plan, 0, -1, kv_out, ws4, stream), "cg_decode (planned)")
        b.record(stream)
        torch.cuda.synchronize()
        cg.check(cg.cg_read_status(ws4), "decode (planned)")
        adaptive = {"level_base": list(lb4), "link": "400 Gb/s, 100 Gb/s from 20 to 45 ms, then 400 Gb/s",
                    "deadline_s": deadline, "levels": lv_plan.tolist(), "total_s": total,
                    "met_deadline": bool(total <= deadline), "fixed_level_total_s": fixed,
                    "container_bytes": n_plan, "assemble_ms": assemble_ms, "decode_ms": a.elapsed_time(b)}
        del tb4, ws4

    # aggregate over ranks: max time, summed bytes
    ms_dec, ms_enc, ms_fit, ms_step_max, ms_e2e, ms_e2e_pipe, ms_e2e_serial = rank_max(
        [ms["dec"], ms["enc"], ms["fit"], ms_step, statistics.mean(e2e_ms), statistics.mean(e2e_pipe_ms),
         statistics.mean(e2e_serial_ms)], world, dev)
    fp16 = w.fp16_bytes
    dec_gbs = job_gbs(nsets * fp16, world, ms_dec)
    enc_gbs = job_gbs(nsets * fp16, world, ms_enc)
    fit_gbs = job_gbs(fp16, world, ms_fit)
    peak, peak_kind = peaks()
    dec_alg = sum(nbytes_list) + nsets * fp16
    enc_alg = nsets * fp16 + sum(nbytes_list)
    dec_ach = dec_alg / (ms["dec"] * 1e-3) / 1e9
    # per step: fit 3 launches, encode 6 per container, decode the index and,
    # at d = 128, one launch per band of chunks per level the range can reach
    dec_launches = 1 + ((1 + (w.n_chunks > 4) + (w.n_chunks > 8)) if w.d == 128 else 1)
    enc_ach = enc_alg / (ms["enc"] * 1e-3) / 1e9
    tb_bytes = tables.numel()

    if world > 1:
        dist.barrier()
    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return
    cpu = None
    if not args.no_cpu_baseline:
        rate, spent, nstreams, rate_enc = cpu_oracle_decode_rate(w, host.numpy().view(np.uint16), budget_s=8.0)
        rate_all, cores = cpu_oracle_decode_rate_all_cores(w.name, budget_s=8.0)
        cpu = {"value": rate_all / 1e9, "unit": "GB/s", "cores": cores, "kind": "oracle",
               "sample": f"oracle decode of chunk streams ({w.C} tokens x {w.d} lanes) of heads spread over the "
                         f"layers, one process per core, 8 s of decode each",
               "single_core": {"value": rate / 1e9, "unit": "GB/s", "cores": 1,
                               "encode_gbs": rate_enc / 1e9,
                               "sample": f"{nstreams} streams, {spent:.1f} s of decode (encode timed apart)"}}
    line = {
        "metric": METRIC, "value": dec_gbs, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step_max, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "u32+f32", "data": "synthetic",
        "config": workload_config(w, world),
        "decode_gbs": dec_gbs, "encode_gbs": enc_gbs, "fit_gbs": fit_gbs,
        "ms": {"fit": ms_fit, "encode": ms_enc, "decode": ms_dec},
        "ratio": fp16 / nbytes, "ratio_incl_tables": fp16 / (nbytes + tb_bytes),
        "container_bytes": nbytes, "tables_bytes": tb_bytes,
        "entropy_bound": {"bound_bytes": ebounds[0], "actual_over_bound": nbytes / ebounds[0] if ebounds[0] else None,
                          "what": "the container against sum over the (layer, K/V, channel) tables of n log2(N/n) "
                                  "/ 8 of its coded symbols + 4 bytes per escape + its structural bytes "
                                  "(cg_entropy_bound, from the fit's histograms); null for a mixed-level container"},
        "per_level": [{"levels": sorted(set(int(v) for v in s_)), "container_bytes": nb_,
                       "ratio": fp16 / nb_, "ratio_incl_tables": fp16 / (nb_ + tb_bytes),
                       "actual_over_bound": nb_ / b_ if b_ else None, "encode_ms": me, "decode_ms": md,
                       "encode_gbs": fp16 / (me * 1e-3) / 1e9, "decode_gbs": fp16 / (md * 1e-3) / 1e9,
                       "decode_frac_of_8TBs": (nb_ + fp16) / (md * 1e-3) / 1e9 / 8000.0}
                      for s_, nb_, b_, me, md in zip(level_sets, nbytes_list, ebounds, ms_enc_sets, ms_dec_sets)],
        "roofline": {"bound": "hbm", "achieved": dec_ach, "peak": peak, "unit": "GB/s", "frac": dec_ach / peak,
                     "traffic": traffic_for("k_decode", fp16), "kernel": "cg_decode",
                     "algorithmic_bytes_per_launch": dec_alg, "peak_kind": peak_kind,
                     "frac_of_8TBs": dec_ach / 8000.0},
        "roofline_encode": {"bound": "hbm", "achieved": enc_ach, "peak": peak, "unit": "GB/s",
                            "frac": enc_ach / peak, "traffic": traffic_for("k_encode", fp16), "kernel": "cg_encode",
                            "algorithmic_bytes_per_launch": enc_alg},
        "e2e": {"value": job_gbs(fp16, world, ms_e2e), "unit": "GB/s", "h2d_bytes_per_step": nbytes,
                "d2h_bytes_per_step": fp16,
                "what": "one cg_decode from a pinned-host container into a pinned-host KV buffer, both mapped "
                        "into the device address space: the decoder reads and writes across the host link",
                "link": dict(link, what="copy-engine rates of the same buffers alone (container in, KV out)",
                             frac_of_d2h_bound=(fp16 / (link["d2h_gbs"] * 1e9)) / (ms_e2e * 1e-3)),
                "pipelined": {"value": job_gbs(fp16, world, ms_e2e_pipe), "unit": "GB/s",
                              "what": "per 4-chunk group: container H2D, cg_decode of the group, strided KV D2H, "
                                      "overlapped with the neighbouring groups on three streams"},
                "serial": {"value": job_gbs(fp16, world, ms_e2e_serial), "unit": "GB/s",
                           "what": "container H2D, one cg_decode, KV D2H, in sequence"}},
        "decode_paged": paged,
        "decode_layer_groups": lgroups,
        "decode_streamed": streamed,
        "adaptive_streaming": adaptive,
        "gpu_launches": args.steps * (3 + nsets * (6 + dec_launches)),
        "clocks": clk,
        "cpu_baseline": cpu,
        "setup": {"generate_s": gen_s},
    }
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
