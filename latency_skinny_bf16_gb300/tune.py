"""Measure every supported plan per (K, N, M) and write the dispatcher's table.

For one call shape, each candidate plan (dot-product with FMA or MMA and each
block_n, split-K with each consumer / cluster size / ring depth / ring chunk)
is forced through the library options and timed L2-cold: a CUDA graph of R
back-to-back calls over R distinct copies of W (together more than 2x the L2
size) is replayed, and the time per call is taken from CUDA events on the
launching stream.  Each candidate is timed twice: with programmatic dependent
launch (consecutive identical calls overlap) and without (each call runs on its
own, as when its neighbours in a decode step are other kernels); the score is
the mean of the two.  The best-scoring plan of each shape becomes one line of
``csrc/tuning_table.inc``; consecutive M with the same winner are merged.

    python -m latency_skinny_bf16_gb300.tune --shapes 7168x256,7168x384 --out table.inc

Shapes are KxN.  Needs a GPU; run it on the machine the table is for.
"""
from __future__ import annotations

import argparse
import json
import math
import sys
import time

import numpy as np
import torch

import latency_skinny_bf16_gb300 as sk

DEFAULT_SHAPES = ["7168x256", "7168x384", "2880x128", "4096x256", "7168x2112", "1536x24576", "14336x7168"]


def token_bucket(M: int) -> int:
    """Kernels are instantiated per token bucket: 1..8, 9..16 (MMA tiles of 8 /
    16 tokens), 17..32 and 33..64 (tensor cores only)."""
    return 8 if M <= 8 else 16 if M <= 16 else 32 if M <= 32 else 64


def tc_candidates(M: int, K: int, N: int, num_sms: int = 152):
    """tcgen05 plans: cluster sizes S along K; for each, the planner's own
    number of row ranges and the range counts that give tiles of about 48 to
    128 rows (W rows come in groups of 8) in one wave of two CTAs per SM; 2 or
    4 boxes per ring stage; the planner's tile height and ring depth."""
    out = []
    G = -(-max(N, 1) // 8)
    for s in (1, 2, 4, 8):
        if K < 2 * s * 128:
            continue
        # one wave at two CTAs per SM (clusters: 90% of the slots, as the planner)
        limit = 2 * num_sms if s == 1 else (2 * num_sms * 9) // (10 * s)
        counts = {0}
        for groups in (6, 8, 12, 16):
            c = -(-G // groups)
            if c <= limit:
                counts.add(c)
        for c in sorted(counts):
            for bk in (128, 256):
                out.append(dict(backend=4, consumer=0, split_k=s, stages=0, block_n=0, stage_k=bk, clusters=c))
    return out


def candidates(M: int, K: int, N: int = 0, num_sms: int = 152):
    out = []
    big = 2 * N * K > 16e6
    if M > 4 or big:
        out += tc_candidates(M, K, N, num_sms)
    if M > 16:
        # 17..64 tokens: tensor cores only -- cluster split-K with the MMA
        # consumer, or the tensor-core dot-product for large weights
        if K % 16:
            return out
        if 2 * N * K > 16e6 and K % 32 == 0:
            for bn in (16, 32, 64):
                out.append(dict(backend=1, consumer=2, split_k=0, stages=0, block_n=bn, stage_k=0))
        for s in (2, 4, 6, 8):
            for bk in (0, 512):           # 0: the dispatcher's ring chunk for this shape
                out.append(dict(backend=2, consumer=2, split_k=s, stages=0, block_n=0, stage_k=bk))
        return out
    for bn in (1, 2, 4, 8):
        out.append(dict(backend=1, block_n=bn, consumer=0, split_k=0, stages=0, stage_k=0))
    if K % 32 == 0:
        for bn in (16, 32, 64):
            out.append(dict(backend=1, block_n=bn, consumer=2, split_k=0, stages=0, stage_k=0))
        # K over a cluster of S CTAs (W by plain loads, DSMEM reduce)
        for s in (2, 4, 8):
            for bn in (16, 32):
                out.append(dict(backend=1, block_n=bn, consumer=2, split_k=s, stages=0, stage_k=0))
    for cons in (1, 2):
        if cons == 2 and K % 16:
            continue
        if big and cons == 2:
            # K-outer streaming: whole K per tile, one CTA per SM
            for bk in (0, 1024, 2048):
                out.append(dict(backend=3, consumer=2, split_k=0, stages=0, block_n=0, stage_k=bk))
        if big:
            for s in (1, 2, 3, 4, 6, 8):
                for bk in (0, 1024, 2048):     # 0: the dispatcher's ring chunk for this shape
                    out.append(dict(backend=2, consumer=cons, split_k=s, stages=0, block_n=0, stage_k=bk))
        else:
            for s in (2, 4, 6, 8):
                for stages in (0, 4):          # 0: the dispatcher's ring depth for this shape
                    out.append(dict(backend=2, consumer=cons, split_k=s, stages=stages, block_n=0, stage_k=0))
    return out


def time_plan(M, N, K, xs, ws, ys, stream, iters=10):
    """us per call: a graph of len(ws) calls over distinct W copies, replayed `iters` times."""
    sh = stream.cuda_stream
    with torch.cuda.stream(stream):
        for x, w, y in zip(xs, ws, ys):
            st = sk.skinny_gemm_bf16(x.data_ptr(), K, w.data_ptr(), K, y.data_ptr(), N, M, N, K, sh)
            if st != sk.SKINNY_OK:
                return None
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        g.capture_begin()
        for x, w, y in zip(xs, ws, ys):
            sk.skinny_gemm_bf16(x.data_ptr(), K, w.data_ptr(), K, y.data_ptr(), N, M, N, K, sh)
        g.capture_end()
    with torch.cuda.stream(stream):
        for _ in range(3):
            g.replay()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(iters):
            g.replay()
        e1.record(stream)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) * 1e3 / (iters * len(ws))


def tune_shape(K, N, m_values, l2_bytes, pdl, log):
    rng = torch.Generator().manual_seed(K * 7919 + N)
    w_bytes = 2 * N * K
    reps = max(4, math.ceil(2 * l2_bytes / w_bytes))
    reps = min(reps, 512)
    w0 = (torch.randn(N, K, generator=rng) * 0.02).to(torch.bfloat16).cuda()
    ws = [w0.clone() for _ in range(reps)]
    stream = torch.cuda.Stream()
    rows = []
    for M in m_values:
        x = torch.randn(M, K, generator=rng).to(torch.bfloat16).cuda()
        xs = [x] * reps
        ys = [torch.empty(M, N, device="cuda") for _ in range(reps)]
        best = None
        results = []
        for c in candidates(M, K, N):
            t0 = time.perf_counter()
            with sk.options(pdl=1, **c):
                try:
                    us_pdl = time_plan(M, N, K, xs, ws, ys, stream)
                except sk.SkinnyError:
                    us_pdl = None
            us_iso = None
            if us_pdl is not None:
                with sk.options(pdl=0, **c):
                    us_iso = time_plan(M, N, K, xs, ws, ys, stream)
            us = None if (us_pdl is None or us_iso is None) else 0.5 * (us_pdl + us_iso)
            wall = time.perf_counter() - t0
            status = sk.skinny_get_device_status()
            log.write(json.dumps({"K": K, "N": N, "M": M, "cand": c, "us": us, "us_pdl": us_pdl, "us_iso": us_iso,
                                  "wall_s": round(wall, 3), "status": status}) + "\n")
            if us is None or status != 0:
                continue
            results.append((us, c))
            if best is None or us < best[0]:
                best = (us, c)
        if best is None:
            # no plan runs this M (e.g. the X slice of 64 tokens does not fit)
            log.write(json.dumps({"K": K, "N": N, "M": M, "best_us": None}) + "\n")
            del ys
            continue
        results.sort(key=lambda t: t[0])
        log.write(json.dumps({"K": K, "N": N, "M": M, "best_us": round(best[0], 3), "best": best[1],
                              "top5": [(round(u, 3), c) for u, c in results[:5]]}) + "\n")
        log.flush()
        rows.append((M, best[1], best[0]))
        del ys
    del ws
    torch.cuda.empty_cache()
    return rows


def merge_rows(K, N, rows, m_max=64):
    """Winners of consecutive tuned M values (in order) that agree -> one table
    line; each line's M range reaches up to the next line's first M, so the
    lines cover every M from the first tuned one to m_max.  A line never
    crosses a token bucket (different kernels, different X footprints), and
    the last line ends with its bucket: untuned buckets keep the default rule."""
    lines = []
    i = 0
    while i < len(rows):
        j = i
        b = token_bucket(rows[i][0])
        while (j + 1 < len(rows) and rows[j + 1][1] == rows[i][1]
               and token_bucket(rows[j + 1][0]) == b):
            j += 1
        c = rows[i][1]
        if j + 1 < len(rows):
            m_hi = min(rows[j + 1][0] - 1, b)
        else:
            m_hi = min(m_max, b)
        lines.append((K, N, rows[i][0], m_hi, c["backend"], c["consumer"], c["split_k"], c["block_n"],
                      c["stages"], c.get("stage_k", 0), c.get("clusters", 0), [round(r[2], 2) for r in rows[i:j + 1]]))
        i = j + 1
    return lines


def plannable_range(K, N, m_lo, m_hi, c, num_sms):
    """The largest m_hi' <= m_hi such that the winner's forced plan exists for
    every M in m_lo..m_hi' (a plan measured at one M may not fit a larger M
    of the same line, e.g. its X slice); M past it keep the default rule."""
    x, w, y = 0x7F0000000000, 0x7F0010000000, 0x7F0020000000   # 16-byte aligned, never dereferenced
    opts = {k: v for k, v in c.items()
            if k in ("backend", "consumer", "split_k", "block_n", "stages", "stage_k", "clusters")}
    last = m_lo - 1
    for M in range(m_lo, m_hi + 1):
        with sk.options(**opts):
            try:
                sk.skinny_plan_for(x, K, w, K, y, N, M, N, K, num_sms)
            except sk.SkinnyError:
                break
        last = M
    return last


def fill_gaps(K, N, lines, num_sms):
    """Token counts left between two lines of a shape (a winner's plan cut short
    by plannable_range) go to the following line, as far down as its plan exists
    (`lines`: (m_lo, m_hi, config) in M order; returns the adjusted list)."""
    x, w, y = 0x7F0000000000, 0x7F0010000000, 0x7F0020000000
    out = []
    for mlo, mhi, c in lines:
        prev_hi = out[-1][1] if out else 0
        if out and mlo > prev_hi + 1 and token_bucket(prev_hi + 1) == token_bucket(mlo):
            opts = {k: v for k, v in c.items()
                    if k in ("backend", "consumer", "split_k", "block_n", "stages", "stage_k", "clusters")}
            while mlo > prev_hi + 1:
                with sk.options(**opts):
                    try:
                        sk.skinny_plan_for(x, K, w, K, y, N, mlo - 1, N, K, num_sms)
                    except sk.SkinnyError:
                        break
                mlo -= 1
        out.append((mlo, mhi, c))
    return out


TABLE = __import__("os").path.join(__import__("os").path.dirname(__file__), "csrc", "tuning_table.inc")


def install(lines, path=TABLE):
    """Write table lines into the compiled-in table: every existing line of a
    tuned (K, N) shape whose M range meets a new line's M range is dropped,
    the new lines take the place of the first dropped one (first match wins in
    the dispatcher), other lines and comments are kept."""
    def parse(line):
        v = [int(x) for x in line.split("//", 1)[0].strip().strip("{},").split(",")]
        return (v[0], v[1]), v[2], v[3]
    new = {}
    for l in lines:
        key, lo, hi = parse(l)
        new.setdefault(key, []).append((lo, hi))
    with open(path) as f:
        old = f.read().rstrip("\n").split("\n")
    out, placed = [], set()
    for l in old:
        if l.strip().startswith("{"):
            key, lo, hi = parse(l)
            if key in new and any(lo <= b and a <= hi for a, b in new[key]):
                if key not in placed:
                    out += [x for x in lines if parse(x)[0] == key]
                    placed.add(key)
                continue
        out.append(l)
    for key in new:
        if key not in placed:
            out += [x for x in lines if parse(x)[0] == key]
    with open(path, "w") as f:
        f.write("\n".join(out) + "\n")


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--shapes", default=",".join(DEFAULT_SHAPES))
    ap.add_argument("--m", default="1-16", help="M values for the router shapes (a-b range or list)")
    ap.add_argument("--m-large", default="1,2,3,4,6,8,9,12,16", help="M values for shapes with W > 16 MB")
    ap.add_argument("--m-mid", default="17,24,32,33,48,64", help="M values 17..64 (split-K MMA), every shape")
    ap.add_argument("--out", default="-")
    ap.add_argument("--install", action="store_true",
                    help="replace the lines of the tuned shapes in csrc/tuning_table.inc with the new ones")
    ap.add_argument("--log", default=None)
    a = ap.parse_args(argv)
    def parse_m(spec):
        if spec in ("", "none"):
            return []
        if "-" in spec:
            lo, hi = (int(v) for v in spec.split("-"))
            return list(range(lo, hi + 1))
        return [int(v) for v in spec.split(",")]
    m_small, m_large, m_mid = parse_m(a.m), parse_m(a.m_large), parse_m(a.m_mid)
    assert sk.skinny_init(0) == sk.SKINNY_OK
    l2 = torch.cuda.get_device_properties(0).L2_cache_size
    log = open(a.log, "a") if a.log else sys.stderr
    out_lines = []
    for shp in a.shapes.split(","):
        K, N = (int(v) for v in shp.lower().split("x"))
        rows = tune_shape(K, N, (m_large if 2 * N * K > 16e6 else m_small) + m_mid, l2, None, log)
        num_sms = torch.cuda.get_device_properties(0).multi_processor_count
        kept = []
        for (k, n, mlo, mhi, be, co, sp, bn, st, bk, cl, us) in merge_rows(K, N, rows):
            c = dict(backend=be, consumer=co, split_k=sp, block_n=bn, stages=st, stage_k=bk, clusters=cl)
            mhi = plannable_range(K, N, mlo, mhi, c, num_sms)
            if mhi >= mlo:
                kept.append((mlo, mhi, dict(c, us=us)))
        for mlo, mhi, c in fill_gaps(K, N, kept, num_sms):
            out_lines.append(f"{{{K}, {N}, {mlo}, {mhi}, {c['backend']}, {c['consumer']}, {c['split_k']}, "
                             f"{c['block_n']}, {c['stages']}, {c['stage_k']}, {c['clusters']}}},  // us/call {c['us']}")
    text = "\n".join(out_lines) + "\n"
    if a.install:
        install(out_lines)
    if a.out == "-":
        sys.stdout.write(text)
    else:
        with open(a.out, "w") as f:
            f.write(text)


if __name__ == "__main__":
    main()
