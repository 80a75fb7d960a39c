"""CPU oracle of the bandwidth-adaptive level controller -- TEST
INFRASTRUCTURE ONLY (the same import rule as the rest of ``oracle/``).

CacheGen adapts each chunk's compression level to the bandwidth available
while a context streams (gptget summary of arXiv 2310.07240, Methodology:
"dynamically adjusting compression according to bandwidth conditions"; the
paper's abstract: raise the compression level when bandwidth drops, to keep
the context-loading delay low).  The pages state no formula.  The reading
used, step by step in plain Python floats (IEEE double, the library's
operation order):

1. Chunks go over one link in order, back to back, starting at time 0.
2. The link is a list of (seconds, bytes_per_s) steps; the last step never
   ends.
3. Before chunk k the bandwidth estimate is the throughput seen on chunk
   k-1 (a given initial estimate for chunk 0).
4. The level is the first l (finest first) such that all remaining chunks
   sent at level l at that estimate leave the last chunk's decode time
   before the deadline; otherwise the last (coarsest) level.
5. Chunk k's decode starts when it has arrived and chunk k-1's decode has
   ended, and lasts decode_s[k].
"""
from __future__ import annotations

import math


def arrival(trace, t0: float, nbytes: float) -> float:
    """Time at which nbytes sent from t0 on have all arrived."""
    if not nbytes > 0.0:
        return t0
    t, rem, step_start = t0, nbytes, 0.0
    for i, (seconds, rate) in enumerate(trace):
        last = i + 1 == len(trace)
        step_end = math.inf if last else step_start + seconds
        if t < step_end:
            cap = math.inf if last else rate * (step_end - t)
            if rem <= cap:
                return t + rem / rate
            rem -= cap
            t = step_end
        step_start = step_end
    return math.inf


def simulate(chunk_bytes, trace, levels, decode_s, choose=False, initial=1.0, deadline=0.0):
    """-> (levels, [(send start, arrival, decode end)], total).  With
    choose=True the levels are picked by rule 4 (``levels`` is ignored)."""
    n, nl = len(chunk_bytes), len(chunk_bytes[0])
    levels = [0] * n if choose else list(levels)
    now, estimate, dec_end = 0.0, initial, 0.0
    tail = decode_s[n - 1]
    timeline = []
    for k in range(n):
        if choose:
            budget = deadline - now - tail
            lv = nl - 1
            for l in range(nl):
                remaining = sum(int(chunk_bytes[j][l]) for j in range(k, n))  # exact integer
                if float(remaining) / estimate <= budget:
                    lv = l
                    break
            levels[k] = lv
        nbytes = float(chunk_bytes[k][levels[k]])
        start = now
        now = arrival(trace, start, nbytes)
        if now > start:
            estimate = nbytes / (now - start)
        dec_end = max(now, dec_end) + decode_s[k]
        timeline.append((start, now, dec_end))
    return levels, timeline, dec_end


def plan(chunk_bytes, trace, initial, deadline, decode_s):
    return simulate(chunk_bytes, trace, None, decode_s, choose=True, initial=initial, deadline=deadline)
