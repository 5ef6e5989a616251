"""GPU parity of the router epilogue (softmax over each token's expert logits
and its top-k) and of the one-call router (GEMM + epilogue), through the C ABI.

The selection compares fp32 logits on both sides (the oracle takes the very
logits the GPU used), so the ids must match exactly; the weights (fp32, CUDA
expf) must satisfy |w - w_ref| <= 1e-5 * w_ref + 1e-9 against the fp64
oracle; and every result is bit-identical from run to run.
"""
import numpy as np
import pytest
import torch

import latency_skinny_bf16_gb300 as sk
import oracle
import skinny_inputs as si
from gpu_util import check_parity, reference

pytestmark = pytest.mark.gpu

W_RTOL, W_ATOL = 1e-5, 1e-9


@pytest.fixture(autouse=True, scope="module")
def _init():
    assert sk.skinny_init(0) == sk.SKINNY_OK
    yield


def check_topk(L: np.ndarray, k: int, renorm: bool, w: np.ndarray, ids: np.ndarray, what=""):
    w_ref, ids_ref = oracle.router_topk(L, k, renormalize=renorm)
    assert np.array_equal(ids, ids_ref), f"{what}: ids differ"
    nan_ref = np.isnan(w_ref)
    assert np.array_equal(np.isnan(w), nan_ref), f"{what}: NaN pattern of the weights differs"
    err = np.abs(w.astype(np.float64)[~nan_ref] - w_ref[~nan_ref])
    bound = W_RTOL * np.abs(w_ref[~nan_ref]) + W_ATOL
    assert (err <= bound).all(), f"{what}: weights off by {err.max():.3e}"


def logits_case(M, N, seed, scale=3.0, ties=False, neg_inf=False):
    rng = np.random.default_rng(seed)
    L = (rng.standard_normal((M, N)) * scale).astype(np.float32)
    if ties:
        L[:, ::4] = np.float32(0.5)
        L[0, 1] = L[0, 2] = L[0, 3] = L[0].max() + 1
    if neg_inf:
        L[:, : N // 2] = -np.inf
    return L


@pytest.mark.parametrize("M,N,k", [(1, 256, 8), (4, 384, 8), (16, 256, 1), (64, 1000, 64), (3, 8192, 16),
                                   (2, 37, 37), (5, 64, 6)])
@pytest.mark.parametrize("renorm", [False, True])
def test_topk_random_logits(M, N, k, renorm):
    L = logits_case(M, N, seed=M * 131 + N + k)
    w, ids = sk.router_topk(torch.from_numpy(L).cuda(), k, renormalize=renorm)
    torch.cuda.synchronize()
    check_topk(L, k, renorm, w.cpu().numpy(), ids.cpu().numpy(), f"M{M} N{N} k{k}")


@pytest.mark.parametrize("kind", ["ties", "neg_inf", "large", "tiny"])
def test_topk_special_rows(kind):
    M, N, k = 8, 256, 16
    if kind == "ties":
        L = logits_case(M, N, 7, ties=True)
    elif kind == "neg_inf":
        L = logits_case(M, N, 8, neg_inf=True)
    elif kind == "large":
        L = logits_case(M, N, 9, scale=300.0)      # most probabilities underflow to 0
    else:
        L = logits_case(M, N, 10, scale=1e-6)      # nearly uniform
    for renorm in (False, True):
        w, ids = sk.router_topk(torch.from_numpy(L).cuda(), k, renormalize=renorm)
        torch.cuda.synchronize()
        check_topk(L, k, renorm, w.cpu().numpy(), ids.cpu().numpy(), kind)


@pytest.mark.parametrize("N", [256, 384, 1000, 2048])
def test_topk_nan_logits(N):
    """NaN logits (at index 0, mid-row, several, a whole row, next to +inf):
    they rank below every other logit, NaNs by index, and the IEEE softmax
    makes every weight of such a row NaN; the ids match the oracle exactly
    and rows without NaN are unaffected.  Both the warp-per-token kernel
    (N <= 1024) and the CTA-per-token kernel run."""
    M, k = 6, 8
    L = logits_case(M, N, seed=4000 + N)
    L[0, 0] = np.nan                                  # first entry
    L[1, N // 2] = np.nan                             # mid-row
    L[2, [1, 5, 9, N - 1]] = np.nan                   # several
    L[3, :] = np.nan                                  # a whole row: ids 0..k-1
    L[4, 3] = np.inf                                  # +inf: inf - inf is NaN
    # row 5 keeps plain values
    for renorm in (False, True):
        w, ids = sk.router_topk(torch.from_numpy(L).cuda(), k, renormalize=renorm)
        torch.cuda.synchronize()
        w, ids = w.cpu().numpy(), ids.cpu().numpy()
        check_topk(L, k, renorm, w, ids, f"NaN rows N{N}")
        assert ids[3].tolist() == list(range(k))
        assert np.isnan(w[:5]).all() and np.isfinite(w[5]).all()
        assert all(len(set(r.tolist())) == k and r.min() >= 0 and r.max() < N for r in ids)


def test_topk_strided_outputs_and_bit_identity():
    M, N, k = 6, 384, 8
    L = logits_case(M, N, 11)
    base = torch.full((M, 400), -5.0, device="cuda")
    base[:, :N] = torch.from_numpy(L).cuda()
    logits = base[:, :N]                                   # ldl = 400
    wbuf = torch.full((M, 13), -7.0, device="cuda")
    ibuf = torch.full((M, 11), -9, dtype=torch.int32, device="cuda")
    first = None
    for _ in range(3):
        w, ids = sk.router_topk(logits, k, renormalize=True, weights=wbuf[:, :k], ids=ibuf[:, :k])
        torch.cuda.synchronize()
        got = (w.cpu().numpy().copy(), ids.cpu().numpy().copy())
        if first is None:
            first = got
            check_topk(L, k, True, *got, "strided")
        else:
            assert np.array_equal(got[0].view(np.uint32), first[0].view(np.uint32))
            assert np.array_equal(got[1], first[1])
    assert (wbuf[:, k:] == -7.0).all() and (ibuf[:, k:] == -9).all()   # gaps untouched


@pytest.mark.parametrize("M", [1, 4, 8, 16, 32])
@pytest.mark.parametrize("N", [256, 384])
def test_router_in_one_call(M, N):
    """GEMM into the caller's logits buffer, then softmax + top-k: the logits
    match the GEMM oracle, the top-k matches the epilogue oracle applied to
    those very logits."""
    case = si.Case(f"router_M{M}_N{N}", M=M, N=N, K=7168, seed=1700 + M + N)
    X, W = si.make_inputs(case)
    x = torch.from_numpy(X.view(np.int16)).cuda()
    w = torch.from_numpy(W.view(np.int16)).cuda()
    k = 8
    logits = torch.empty((M, N), dtype=torch.float32, device="cuda")
    wt = torch.empty((M, k), dtype=torch.float32, device="cuda")
    ids = torch.empty((M, k), dtype=torch.int32, device="cuda")
    for pdl in (0, 1):
        with sk.options(pdl=pdl):
            st = sk.skinny_router_bf16_topk(x.data_ptr(), 7168, w.data_ptr(), 7168, logits.data_ptr(), N, M, N,
                                            7168, k, 1, wt.data_ptr(), k, ids.data_ptr(), k, 0)
        assert st == sk.SKINNY_OK
        torch.cuda.synchronize()
        L = logits.cpu().numpy()
        yref, A = reference(case, X, W)
        check_parity(L, yref, A, case.name)
        check_topk(L, k, True, wt.cpu().numpy(), ids.cpu().numpy(), case.name)
    assert sk.skinny_get_device_status() == 0


@pytest.mark.parametrize("pdl", [0, 1])
def test_router_graph_chain_matches_eager(pdl):
    """Several one-call routers captured in one CUDA graph reproduce the eager
    results bit for bit (with PDL each epilogue overlaps its GEMM's tail)."""
    cfgs = [(4, 256), (16, 384), (8, 256)]
    bufs = []
    for i, (M, N) in enumerate(cfgs):
        case = si.Case(f"rg{i}", M=M, N=N, K=7168, seed=1800 + i)
        X, W = si.make_inputs(case)
        bufs.append(dict(M=M, N=N, x=torch.from_numpy(X.view(np.int16)).cuda(),
                         w=torch.from_numpy(W.view(np.int16)).cuda(),
                         L=torch.empty((M, N), device="cuda"), wt=torch.empty((M, 8), device="cuda"),
                         ids=torch.empty((M, 8), dtype=torch.int32, device="cuda")))

    def launch(s):
        for b in bufs:
            assert sk.skinny_router_bf16_topk(b["x"].data_ptr(), 7168, b["w"].data_ptr(), 7168, b["L"].data_ptr(),
                                              b["N"], b["M"], b["N"], 7168, 8, 0, b["wt"].data_ptr(), 8,
                                              b["ids"].data_ptr(), 8, s) == sk.SKINNY_OK
    with sk.options(pdl=pdl):
        s = torch.cuda.Stream()
        with torch.cuda.stream(s):
            launch(s.cuda_stream)
        torch.cuda.synchronize()
        eager = [(b["wt"].cpu().clone(), b["ids"].cpu().clone()) for b in bufs]
        for b in bufs:
            b["wt"].zero_()
            b["ids"].zero_()
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            launch(s.cuda_stream)
        for _ in range(3):
            g.replay()
        torch.cuda.synchronize()
    for b, (we, ie) in zip(bufs, eager):
        assert torch.equal(b["wt"].cpu().view(torch.int32), we.view(torch.int32))
        assert torch.equal(b["ids"].cpu(), ie)
