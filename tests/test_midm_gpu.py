"""GPU parity of the medium-M path (17..64 tokens on the tensor cores: cluster
split-K with the mma.sync consumer, the tensor-core dot-product, tcgen05)
against the oracle, through the C ABI.

Same bar as the M <= 16 tests: |y - y_ref| <= 1e-5 * sum_k |x*w| + 1e-6,
cosine >= 0.99999, nothing written outside Y[:M, :N], bit-identical runs.
"""
import numpy as np
import pytest
import torch

import latency_skinny_bf16_gb300 as sk
import skinny_inputs as si
from gpu_util import Buffers, check_parity, reference, run_and_check

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True, scope="module")
def _init():
    assert sk.skinny_init(0) == sk.SKINNY_OK
    yield


def _ids(cases):
    return [c.name for c in cases]


MIDM = si.midm_cases()


@pytest.mark.parametrize("case", MIDM, ids=_ids(MIDM))
def test_midm_workload_and_bit_identity(case):
    X, W = si.make_inputs(case)
    b = Buffers(case, X, W)
    p = b.plan()
    assert p["consumer"] == sk.SKINNY_CONSUMER_MMA      # tensor cores only
    yref, A = reference(case, X, W)
    first = None
    for _ in range(3):
        assert b.run() == sk.SKINNY_OK
        y = b.y_mat().copy()
        if first is None:
            first = y
            check_parity(y, yref, A, case.name)
        else:
            assert np.array_equal(y.view(np.uint32), first.view(np.uint32)), "run-to-run bits differ"
    assert b.canary_ok()
    assert sk.skinny_get_device_status() == 0


MIDM_EDGE = si.midm_edge_cases()


@pytest.mark.parametrize("chunk", range(4))
def test_midm_edge_cases(chunk):
    for case in MIDM_EDGE[chunk * 10:(chunk + 1) * 10]:
        run_and_check(case)
    assert sk.skinny_get_device_status() == 0


# forced split sizes / ring depths / chunk lengths, ragged N and K tails
FORCED_MIDM = [
    si.Case("fm_m17", M=17, N=37, K=4096, seed=451),
    si.Case("fm_m24", M=24, N=100, K=1040, seed=452),      # K % 64 != 0: ragged last chunk
    si.Case("fm_m33", M=33, N=16, K=2880, seed=453),
    si.Case("fm_m64", M=64, N=130, K=7168, seed=454, w_dist="uniform_isqrtk"),
    si.Case("fm_k16", M=40, N=19, K=16, seed=455),         # one k16 step
]


def _midm_variants():
    out = []
    for s in (1, 2, 3, 8):
        for stages in (1, 2, 4):
            for stage_k in (0, 256):
                out.append(dict(backend=sk.SKINNY_BACKEND_SPLITK, consumer=sk.SKINNY_CONSUMER_MMA,
                                split_k=s, stages=stages, stage_k=stage_k))
    return out


@pytest.mark.parametrize("case", FORCED_MIDM, ids=_ids(FORCED_MIDM))
def test_midm_every_variant(case):
    X, W = si.make_inputs(case)
    yref, A = reference(case, X, W)
    ran = 0
    for v in _midm_variants():
        with sk.options(**v):
            b = Buffers(case, X, W, ldy=case.N + 5)
            st = b.run()
            if st == sk.SKINNY_ERR_UNSUPPORTED:
                with pytest.raises(sk.SkinnyError):   # refused on the host, like the planner says
                    b.plan()
                continue
            assert st == sk.SKINNY_OK, (v, sk.skinny_status_string(st))
            check_parity(b.y_mat(), yref, A, f"{case.name} {v}")
            assert b.canary_ok(), v
            assert sk.skinny_get_device_status() == 0, v
            ran += 1
    # 64 tokens at K = 7168 fit only the larger clusters (the X slice must fit shared memory)
    assert ran >= (len(_midm_variants()) // 2 if case.M <= 32 else len(_midm_variants()) // 4)


@pytest.mark.parametrize("ldx_pad,x_off", [(0, 0), (8, 0), (3, 0), (0, 1)])
@pytest.mark.parametrize("M", [17, 64])
def test_midm_x_strides_and_misalignment(ldx_pad, x_off, M):
    """X with row padding, rows that are not 16-byte aligned (staged by the
    consumer warps instead of bulk copies), and an odd base offset."""
    case = si.Case(f"midm_x_{M}_{ldx_pad}_{x_off}", M=M, N=256, K=4096, seed=460 + ldx_pad + x_off)
    run_and_check(case, ldx=case.K + ldx_pad, x_offset=x_off)


def test_midm_rows_do_not_depend_on_other_tokens():
    """Within one token bucket (33..64 share a kernel) and one plan, the first
    rows of a 64-token call are bit-identical to a 40-token call on the same
    rows: tokens never mix."""
    big = si.Case("midm_rows64", M=64, N=384, K=4096, seed=470)
    X, W = si.make_inputs(big)
    small = si.Case("midm_rows40", M=40, N=384, K=4096, seed=470)
    with sk.options(backend=sk.SKINNY_BACKEND_SPLITK, consumer=sk.SKINNY_CONSUMER_MMA, split_k=8, stages=2):
        b64 = Buffers(big, X, W)
        b40 = Buffers(small, X[:40].copy(), W)
        assert b64.run() == sk.SKINNY_OK and b40.run() == sk.SKINNY_OK
        y64, y40 = b64.y_mat(), b40.y_mat()
    assert np.array_equal(y64[:40].view(np.uint32), y40.view(np.uint32))


def test_midm_bf16_output():
    case = si.Case("midm_bf16", M=48, N=2112, K=7168, seed=480, w_dist="uniform_isqrtk")
    X, W = si.make_inputs(case)
    yref, A = reference(case, X, W)
    x = torch.from_numpy(X.view(np.int16)).cuda().view(torch.bfloat16)
    w = torch.from_numpy(W.view(np.int16)).cuda().view(torch.bfloat16)
    y32 = sk.gemm(x, w)
    y16 = torch.empty(case.M, case.N, dtype=torch.bfloat16, device="cuda")
    sk.gemm(x, w, out=y16)
    torch.cuda.synchronize()
    check_parity(y32.cpu().numpy(), yref, A, case.name)
    # the bf16 result is the fp32 result rounded to nearest-even, bit for bit
    assert torch.equal(y16.cpu(), y32.cpu().to(torch.bfloat16))


@pytest.mark.parametrize("pdl", [0, 1])
def test_midm_graph_capture_chain(pdl):
    """A chain of mid-M calls captured in a CUDA graph, with and without PDL,
    reproduces the eager results bit for bit."""
    cases = [si.Case(f"midm_g{i}", M=M, N=N, K=K, seed=490 + i)
             for i, (M, N, K) in enumerate([(17, 256, 7168), (64, 384, 4096), (32, 2112, 7168)])]
    with sk.options(pdl=pdl):
        bufs = [Buffers(c, *si.make_inputs(c)) for c in cases]
        s = torch.cuda.Stream()
        with torch.cuda.stream(s):
            for b in bufs:
                assert b.run(s.cuda_stream) == sk.SKINNY_OK
        torch.cuda.synchronize()
        eager = [b.y_mat().copy() for b in bufs]
        for b in bufs:
            b.y_dev.fill_(0.0)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            for b in bufs:
                assert b.run(s.cuda_stream) == sk.SKINNY_OK
        for _ in range(3):
            g.replay()
        torch.cuda.synchronize()
    for b, e, c in zip(bufs, eager, cases):
        assert np.array_equal(b.y_mat().view(np.uint32), e.view(np.uint32)), c.name
    assert sk.skinny_get_device_status() == 0


@pytest.mark.parametrize("bn", [16, 32, 64])
@pytest.mark.parametrize("M", [17, 24, 33, 64])
def test_midm_tensor_core_dotprod(M, bn):
    """17..64 tokens on the tensor-core dot-product (the route for large
    weights): ragged N, X staged in several chunks, strided Y."""
    for i, (N, K) in enumerate([(130, 1536), (100, 14336), (300, 4096)]):
        case = si.Case(f"midm_dm_M{M}_bn{bn}_{N}_{K}", M=M, N=N, K=K, seed=3400 + 10 * M + bn + i,
                       w_dist="uniform_isqrtk", ldy=N + 3)
        X, W = si.make_inputs(case)
        with sk.options(backend=sk.SKINNY_BACKEND_DOTPROD, consumer=sk.SKINNY_CONSUMER_MMA, block_n=bn):
            b = Buffers(case, X, W)
            p = b.plan()
            assert (p["backend"], p["consumer"], p["block_n"]) == (sk.SKINNY_BACKEND_DOTPROD,
                                                                   sk.SKINNY_CONSUMER_MMA, bn)
            yref, A = reference(case, X, W)
            first = None
            for _ in range(2):
                assert b.run() == sk.SKINNY_OK
                y = b.y_mat().copy()
                if first is None:
                    first = y
                    check_parity(y, yref, A, case.name)
                else:
                    assert np.array_equal(y.view(np.uint32), first.view(np.uint32))
            assert b.canary_ok()
    assert sk.skinny_get_device_status() == 0
