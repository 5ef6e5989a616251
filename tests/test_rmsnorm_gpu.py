"""GPU parity of the q_b projection with its query RMS norm in front
(skinny_rmsnorm_gemm_bf16) against the oracle.

The stored XN is a bf16 rounding of x * r * g computed in fp32; the oracle
gives that value in fp64.  Each XN element must be the nearest bf16 of the
oracle's value, except where the fp32 computation may land on the other side
of a rounding midpoint: within the relative distance `xn_allowance(K)` of it,
derived below from the kernel's arithmetic, either neighbour is correct.  Y
must match the GEMM oracle applied to the XN the GPU produced (the standard
tolerance), and everything is bit-identical run to run and with PDL on or off.
"""
import math

import numpy as np
import pytest
import torch

import latency_skinny_bf16_gb300 as sk
import oracle
import skinny_inputs as si
from gpu_util import check_parity

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True, scope="module")
def _init():
    assert sk.skinny_init(0) == sk.SKINNY_OK
    yield


def bf16_to_f64(bits):
    return (np.asarray(bits, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


U = 2.0 ** -24          # fp32 unit roundoff


def xn_allowance(K: int) -> float:
    """Relative error bound of the fp32 value x * r * g before its rounding to bf16.

    The norm kernel sums the K squares of a token with 128 threads: thread j
    adds, in order, the squares of the elements of its 8-element chunks
    c = j, j + 128, ... (one fused multiply-add each; a bf16 square is exact in
    fp32), then a 5-level warp butterfly and the 4 warps in order.  The longest
    chain of rounded adds is L = 8 * ceil(K / 1024) + 5 + 3, and every term is
    non-negative, so the sum t' = t (1 + a) with |a| <= gamma_L = L u / (1 - L u).
    Then, to first order in u:
      q = t' / K (one rounding), + eps (eps itself rounded to fp32, one
      rounding of the add):                       gamma_L + 2u
      s = sqrt(.) halves that and rounds once:    gamma_L / 2 + 2u
      r = 1 / s:                                  gamma_L / 2 + 3u
      (x * r) * g, two roundings:                 gamma_L / 2 + 5u
    The factor 1.001 covers the second-order terms (products of two or more
    of the u-sized errors, below 1e-12 here)."""
    L = 8 * math.ceil(K / 1024) + 8
    gamma = L * U / (1 - L * U)
    return 1.001 * (gamma / 2 + 5 * U)


def bf16_rne(v: np.ndarray) -> np.ndarray:
    """Nearest bf16 (ties to even) of float64 values, rounded once (no fp32
    step): v = m * 2^e with 0.5 <= |m| < 1, and bf16 keeps 8 significant bits."""
    m, e = np.frexp(v)
    return np.ldexp(np.round(m * 256.0) / 256.0, e)   # np.round: ties to even


def check_xn(xn_bits, ref, K):
    """xn_bits (bf16) against the unrounded fp64 reference values: the nearest
    bf16, or its neighbour when the reference lies within xn_allowance(K)
    (relative) of the midpoint between them."""
    got = bf16_to_f64(xn_bits)
    rn = bf16_rne(ref)
    ok = got == rn
    if not ok.all():
        bad = ~ok
        v = ref[bad]
        mid = 0.5 * (got[bad] + rn[bad])
        near_mid = np.abs(v - mid) <= xn_allowance(K) * np.abs(v)
        # got is the other neighbour: one bf16 step (2^-7 of the binade) away
        adjacent = np.abs(got[bad] - rn[bad]) <= np.abs(v) * 2.0 ** -7 * 1.0001
        assert (near_mid & adjacent).all(), f"{int((~(near_mid & adjacent)).sum())} XN elements off"
    return float((~ok).mean())


def make_case(M, N, K, seed):
    case = si.Case(f"qb_M{M}_N{N}_K{K}", M=M, N=N, K=K, seed=seed, w_dist="uniform_isqrtk")
    X, W = si.make_inputs(case)
    g = torch.Generator().manual_seed(seed + 17)
    G = si._to_bf16_bits(1.0 + 0.1 * torch.randn(K, generator=g))
    return case, X, W, G


def run_norm(case, X, W, G, eps=1e-6, ldx=None, pdl=None):
    M, N, K = case.M, case.N, case.K
    ldx = ldx or K
    x = torch.from_numpy(si.embed_rows(X, ldx).view(np.int16).copy()).cuda()
    w = torch.from_numpy(W.view(np.int16)).cuda()
    gd = torch.from_numpy(G.view(np.int16)).cuda()
    xn = torch.zeros(M * K + 8, dtype=torch.int16, device="cuda")
    y = torch.full((M * N + 8,), -7.0, device="cuda")
    opts = {} if pdl is None else dict(pdl=pdl)
    with sk.options(**opts):
        st = sk.skinny_rmsnorm_gemm_bf16(x.data_ptr(), ldx, gd.data_ptr(), eps, xn.data_ptr(), K, w.data_ptr(), K,
                                         y.data_ptr(), N, M, N, K, 0)
    assert st == sk.SKINNY_OK
    torch.cuda.synchronize()
    xn_bits = xn.cpu().numpy()[: M * K].view(np.uint16).reshape(M, K)
    yv = y.cpu().numpy()
    assert (yv[M * N:] == -7.0).all()
    return xn_bits, yv[: M * N].reshape(M, N)


@pytest.mark.parametrize("M", [1, 2, 3, 8, 16, 32])
def test_qb_projection_with_norm(M):
    case, X, W, G = make_case(M, 24576, 1536, seed=3000 + M)
    xn_bits, y = run_norm(case, X, W, G)
    frac = check_xn(xn_bits, oracle.rmsnorm(X, G, 1e-6, M, 1536), 1536)
    assert frac < 1e-3
    yref, A = oracle.gemm(xn_bits, W, M, 24576, 1536)
    check_parity(y, yref, A, case.name)
    assert sk.skinny_get_device_status() == 0


@pytest.mark.parametrize("backend", [dict(backend=1), dict(backend=1, consumer=2, block_n=32),
                                     dict(backend=2, consumer=2, split_k=4), dict(backend=2, consumer=1),
                                     dict(backend=3)])
def test_norm_reaches_every_backend(backend):
    """Whichever backend runs the GEMM, it reads XN only after the norm finished
    (PDL on), and the result equals the no-PDL run bit for bit."""
    case, X, W, G = make_case(8, 2112, 1536, seed=3100)
    with sk.options(**backend):
        xa, ya = run_norm(case, X, W, G, pdl=1)
        xb, yb = run_norm(case, X, W, G, pdl=0)
    assert np.array_equal(xa, xb) and np.array_equal(ya.view(np.uint32), yb.view(np.uint32))
    check_xn(xa, oracle.rmsnorm(X, G, 1e-6, 8, 1536), 1536)
    yref, A = oracle.gemm(xa, W, 8, 2112, 1536)
    check_parity(ya, yref, A, f"norm + {backend}")


def test_norm_strided_x_eps_and_ragged_k():
    case, X, W, G = make_case(5, 130, 1000, seed=3200)
    for eps in (0.0, 1e-6, 0.5):
        xn_bits, y = run_norm(case, X, W, G, eps=eps, ldx=1003)
        check_xn(xn_bits, oracle.rmsnorm(X, G, eps, 5, 1000), 1000)
        yref, A = oracle.gemm(xn_bits, W, 5, 130, 1000)
        check_parity(y, yref, A, f"eps={eps}")


def test_norm_wrapper_and_graph():
    case, X, W, G = make_case(4, 24576, 1536, seed=3300)
    x = torch.from_numpy(X.view(np.int16)).cuda().view(torch.bfloat16)
    w = torch.from_numpy(W.view(np.int16)).cuda().view(torch.bfloat16)
    g = torch.from_numpy(G.view(np.int16)).cuda().view(torch.bfloat16)
    y, xn = sk.rmsnorm_gemm(x, g, 1e-6, w)
    torch.cuda.synchronize()
    for pdl in (0, 1):
        with sk.options(pdl=pdl):
            s = torch.cuda.Stream()
            y2 = torch.zeros_like(y)
            xn2 = torch.zeros_like(xn)
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph, stream=s):
                sk.rmsnorm_gemm(x, g, 1e-6, w, out=y2, xn=xn2, stream=s)
            graph.replay()
            torch.cuda.synchronize()
        assert torch.equal(y2.view(torch.int32), y.view(torch.int32)) and torch.equal(xn2, xn)


# ---------------------------------------------------------------- the fused form (one launch)

FUSED_CASES = [
    # (M, N, K, tcgen05 plan options)
    (1, 24576, 1536, {}),
    (3, 24576, 1536, {}),
    (8, 2112, 1536, {}),
    (16, 24576, 1536, {}),
    (16, 2112, 1536, dict(split_k=1, clusters=33)),
    (12, 300, 1536, dict(split_k=1, stage_k=64)),
    (7, 1000, 1000, {}),                       # K % 64 != 0: the last box is part zeros
    (16, 520, 520, dict(split_k=1, stage_k=128)),
    (16, 2112, 1536, dict(split_k=2)),         # K split over a cluster: the two-launch form
]


@pytest.mark.parametrize("M,N,K,opts", FUSED_CASES, ids=[f"M{m}_N{n}_K{k}_{o}" for m, n, k, o in FUSED_CASES])
def test_fused_norm_equals_two_launches(M, N, K, opts):
    """The norm inside the tcgen05 GEMM (one launch) gives the same XN bits as
    the norm kernel, and, under the same plan, the same Y bits as the norm
    kernel followed by the GEMM; both match the oracle."""
    case, X, W, G = make_case(M, N, K, seed=3400 + M + N % 97 + K)
    with sk.options(backend=sk.SKINNY_BACKEND_TCGEN05, **opts):
        with sk.options(fuse_norm=1):
            xf, yf = run_norm(case, X, W, G)
        with sk.options(fuse_norm=0):
            xs, ys = run_norm(case, X, W, G)
    assert np.array_equal(xf, xs), "XN differs between the fused and the two-launch forms"
    assert np.array_equal(yf.view(np.uint32), ys.view(np.uint32)), "Y differs between the two forms"
    check_xn(xf, oracle.rmsnorm(X, G, 1e-6, M, K), K)
    cols = np.arange(N) if N <= 2112 else np.sort(np.random.default_rng(M).choice(N, 1024, replace=False))
    yref, A = oracle.gemm(xf, np.ascontiguousarray(W[cols]), M, len(cols), K)
    check_parity(yf[:, cols], yref, A, f"fused M{M} N{N} K{K}")
    assert sk.skinny_get_device_status() == 0


def test_fused_norm_timeout_path_reports_and_recovers():
    """A wait budget of 0 on the fused form: its waits (raw X landed, X
    normalised, ring stages, accumulators) give up at once and are reported;
    the CTA still lets its copies land (bounded), passes its barriers, frees
    tensor memory once its MMAs are done and exits.  The next call is exact."""
    case, X, W, G = make_case(8, 640, 1536, seed=3600)
    assert sk.skinny_get_device_status() == 0
    with sk.options(backend=sk.SKINNY_BACKEND_TCGEN05, fuse_norm=1, wait_timeout_us=0):
        run_norm(case, X, W, G)
        code = sk.skinny_get_device_status()
    assert code & 0xFF == sk.SKINNY_ERR_DEVICE_TIMEOUT
    assert sk.skinny_get_device_status() == 0
    with sk.options(backend=sk.SKINNY_BACKEND_TCGEN05, fuse_norm=1):
        xf, yf = run_norm(case, X, W, G)
    check_xn(xf, oracle.rmsnorm(X, G, 1e-6, 8, 1536), 1536)
    yref, A = oracle.gemm(xf, W, 8, 640, 1536)
    check_parity(yf, yref, A, "fused norm after a timeout")
    assert sk.skinny_get_device_status() == 0


def test_fused_norm_strided_and_misaligned_x_and_eps():
    """Strided X rows (16-byte aligned: the fused form; not aligned: the
    two-launch form) and several eps: both forms give the same bits."""
    case, X, W, G = make_case(5, 640, 1000, seed=3500)
    for eps, ldx in ((0.0, 1008), (1e-6, 1003), (0.5, 1016)):
        with sk.options(backend=sk.SKINNY_BACKEND_TCGEN05):
            with sk.options(fuse_norm=1):
                xf, yf = run_norm(case, X, W, G, eps=eps, ldx=ldx)
            with sk.options(fuse_norm=0):
                xs, ys = run_norm(case, X, W, G, eps=eps, ldx=ldx)
        assert np.array_equal(xf, xs) and np.array_equal(yf.view(np.uint32), ys.view(np.uint32)), eps
        check_xn(xf, oracle.rmsnorm(X, G, eps, 5, 1000), 1000)


@pytest.mark.parametrize("pdl", [0, 1])
def test_fused_norm_in_a_graph_chain(pdl):
    """Two fused calls back to back in a CUDA graph (the second reads nothing
    the first writes), replayed: the same bits as eager calls."""
    cases = [make_case(16, 24576, 1536, seed=3600), make_case(4, 2112, 1536, seed=3601)]
    with sk.options(pdl=pdl, fuse_norm=1):
        eager = [run_norm(*c) for c in cases]
        tens = []
        for case, X, W, G in cases:
            M, N, K = case.M, case.N, case.K
            tens.append(dict(x=torch.from_numpy(X.view(np.int16).copy()).cuda(),
                             w=torch.from_numpy(W.view(np.int16)).cuda(),
                             g=torch.from_numpy(G.view(np.int16)).cuda(),
                             xn=torch.zeros(M * K, dtype=torch.int16, device="cuda"),
                             y=torch.zeros(M * N, device="cuda"), M=M, N=N, K=K))
        s = torch.cuda.Stream()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=s):
            for t in tens:
                st = sk.skinny_rmsnorm_gemm_bf16(t["x"].data_ptr(), t["K"], t["g"].data_ptr(), 1e-6,
                                                 t["xn"].data_ptr(), t["K"], t["w"].data_ptr(), t["K"],
                                                 t["y"].data_ptr(), t["N"], t["M"], t["N"], t["K"], s.cuda_stream)
                assert st == sk.SKINNY_OK
        for _ in range(3):
            graph.replay()
        torch.cuda.synchronize()
    for t, (xe, ye) in zip(tens, eager):
        assert np.array_equal(t["xn"].cpu().numpy().view(np.uint16).reshape(xe.shape), xe)
        assert np.array_equal(t["y"].cpu().numpy().reshape(ye.shape).view(np.uint32), ye.view(np.uint32))
    assert sk.skinny_get_device_status() == 0
