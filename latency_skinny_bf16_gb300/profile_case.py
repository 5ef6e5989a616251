"""Run one call shape of one kernel family a few times, for a profiler.

    python -m latency_skinny_bf16_gb300.profile_case --kernel tmem_gemm --M 16 --N 24576 --K 1536 --launches 3

The family is forced through the library options (the dispatcher's own plan
for the shape when ``--kernel auto``); ``--warmup`` untimed launches come
first, then ``--launches`` launches, each on its own copy of W (together more
than 2x the L2 size when ``--cold``), so a profiler capturing the last
launches sees DRAM traffic, not L2 hits.  The router epilogue (``topk``), the
query RMS norm in front of the q_b projection (``rmsnorm``: the norm kernel
and the GEMM behind it) and the fp32-weight router (``f32w``) run through
their own entry points.  Prints the plan of the call.
"""
from __future__ import annotations

import argparse
import json
import math

import torch

import latency_skinny_bf16_gb300 as sk

FAMILIES = {
    "auto": {},
    "dotprod": dict(backend=sk.SKINNY_BACKEND_DOTPROD, consumer=sk.SKINNY_CONSUMER_FMA),
    "dotmma": dict(backend=sk.SKINNY_BACKEND_DOTPROD, consumer=sk.SKINNY_CONSUMER_MMA),
    "splitk": dict(backend=sk.SKINNY_BACKEND_SPLITK),
    "stream": dict(backend=sk.SKINNY_BACKEND_STREAM),
    "tmem_gemm": dict(backend=sk.SKINNY_BACKEND_TCGEN05),
}


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--kernel", default="auto",
                    choices=sorted(FAMILIES) + ["topk", "rmsnorm", "f32w"])
    ap.add_argument("--M", type=int, default=16)
    ap.add_argument("--N", type=int, default=24576)
    ap.add_argument("--K", type=int, default=1536)
    ap.add_argument("--k", type=int, default=8, help="experts chosen (topk)")
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--launches", type=int, default=3)
    ap.add_argument("--cold", action="store_true", help="distinct W copies totalling more than 2x L2")
    ap.add_argument("--pdl", type=int, default=0, choices=[0, 1])
    ap.add_argument("--split-k", type=int, default=0, help="force the K split (0: the family's own)")
    ap.add_argument("--block-n", type=int, default=0, help="force block_n (0: the family's own)")
    ap.add_argument("--fuse", type=int, default=1, choices=[0, 1],
                    help="rmsnorm: 1 = the norm inside the tcgen05 GEMM when the plan allows, 0 = two launches")
    a = ap.parse_args(argv)
    assert sk.skinny_init(0) == sk.SKINNY_OK
    M, N, K = a.M, a.N, a.K
    g = torch.Generator().manual_seed(1234)
    n_calls = a.warmup + a.launches
    l2 = torch.cuda.get_device_properties(0).L2_cache_size
    wdt = torch.float32 if a.kernel == "f32w" else torch.bfloat16
    w_bytes = N * K * (4 if a.kernel == "f32w" else 2)
    copies = max(1, min(n_calls, math.ceil(2 * l2 / max(w_bytes, 1)))) if a.cold else 1
    w0 = (torch.rand(N, K, generator=g) * 2 - 1).div(math.sqrt(K)).to(wdt).cuda()
    ws = [w0] + [w0.clone() for _ in range(copies - 1)]
    x = torch.randn(M, K, generator=g).to(torch.bfloat16).cuda()
    y = torch.empty(M, N, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    plan = None
    forced = dict(FAMILIES.get(a.kernel, {}))
    if a.split_k:
        forced["split_k"] = a.split_k
    if a.block_n:
        forced["block_n"] = a.block_n
    with sk.options(pdl=a.pdl, fuse_norm=a.fuse, **forced):
        for i in range(n_calls):
            w = ws[i % copies]
            if a.kernel == "topk":
                logits = torch.randn(M, N, generator=g).cuda() if i == 0 else logits
                wt = torch.empty(M, a.k, device="cuda")
                ids = torch.empty(M, a.k, dtype=torch.int32, device="cuda")
                st = sk.skinny_router_topk(logits.data_ptr(), N, M, N, a.k, 0, wt.data_ptr(), a.k, ids.data_ptr(),
                                           a.k, s)
            elif a.kernel == "rmsnorm":
                gamma = (1 + 0.1 * torch.randn(K, generator=g)).to(torch.bfloat16).cuda() if i == 0 else gamma
                xn = torch.empty_like(x)
                st = sk.skinny_rmsnorm_gemm_bf16(x.data_ptr(), K, gamma.data_ptr(), 1e-6, xn.data_ptr(), K,
                                                 w.data_ptr(), K, y.data_ptr(), N, M, N, K, s)
            elif a.kernel == "f32w":
                st = sk.skinny_gemm_bf16_f32w(x.data_ptr(), K, w.data_ptr(), K, y.data_ptr(), N, M, N, K, s)
                if plan is None:
                    plan = sk.skinny_plan_for_f32w(x.data_ptr(), K, w.data_ptr(), K, y.data_ptr(), N, M, N, K,
                                                   torch.cuda.get_device_properties(0).multi_processor_count)
            else:
                st = sk.skinny_gemm_bf16(x.data_ptr(), K, w.data_ptr(), K, y.data_ptr(), N, M, N, K, s)
                if plan is None:
                    plan = sk.skinny_query_plan(x.data_ptr(), K, w.data_ptr(), K, y.data_ptr(), N, M, N, K)
            if st != sk.SKINNY_OK:
                raise sk.SkinnyError(st, a.kernel)
        torch.cuda.synchronize()
    code = sk.skinny_get_device_status()
    if code:
        raise RuntimeError(f"device status {code:#x}")
    print(json.dumps({"kernel": a.kernel, "M": M, "N": N, "K": K, "plan": plan, "w_copies": copies,
                      "algorithmic_bytes": 2 * N * K * (2 if a.kernel == "f32w" else 1) + 2 * M * K + 4 * M * N}))


if __name__ == "__main__":
    main()
