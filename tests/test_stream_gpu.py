"""GPU parity of the K-outer streaming backend (one CTA per SM, whole K per
16-row tile, X and W through one ring chunk by chunk) against the oracle,
through the C ABI.

Same bar as the other kernels: |y - y_ref| <= 1e-5 * sum_k |x*w| + 1e-6,
cosine >= 0.99999, nothing written outside Y[:M, :N], bit-identical runs.
"""
import numpy as np
import pytest
import torch

import latency_skinny_bf16_gb300 as sk
import skinny_inputs as si
from gpu_util import Buffers, check_parity, reference, run_and_check

pytestmark = pytest.mark.gpu

STREAM = dict(backend=sk.SKINNY_BACKEND_STREAM)


@pytest.fixture(autouse=True, scope="module")
def _init():
    assert sk.skinny_init(0) == sk.SKINNY_OK
    yield


def _ids(cases):
    return [c.name for c in cases]


# the projection shapes the backend is for, at every token bucket
PROJ = [si.Case(f"st_M{M}_N{N}_K{K}", M=M, N=N, K=K, seed=1000 + i, w_dist="uniform_isqrtk", ldy=N + 64)
        for i, (M, N, K) in enumerate([(2, 7168, 14336), (8, 7168, 14336), (16, 7168, 14336),
                                       (3, 2112, 7168), (9, 2112, 7168), (16, 2112, 7168)])]


@pytest.mark.parametrize("case", PROJ, ids=_ids(PROJ))
def test_stream_projection_shapes_and_bit_identity(case):
    X, W = si.make_inputs(case)
    yref, A = reference(case, X, W)
    with sk.options(**STREAM):
        b = Buffers(case, X, W)
        assert b.plan()["backend"] == sk.SKINNY_BACKEND_STREAM
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


# ragged N and K, several tiles per CTA, the smallest legal ring, short chunks
FORCED = [
    si.Case("sf_ragged", M=3, N=16 * 13 + 5, K=4096, seed=1101),
    si.Case("sf_ktail", M=16, N=37, K=1040, seed=1102),        # K % 64 == 16: a short last chunk
    si.Case("sf_k2880", M=9, N=130, K=2880, seed=1103),
    si.Case("sf_k16", M=5, N=19, K=16, seed=1104),            # one k16 step
    si.Case("sf_m1", M=1, N=100, K=7168, seed=1105),
    si.Case("sf_outl", M=8, N=64, K=8192, seed=1106, x_dist="normal", w_dist="normal", outliers=True),
]


def _variants(case):
    tiles = -(-case.N // 16)
    out = []
    for ctas in sorted({0, max(1, -(-tiles // 4)), max(1, -(-tiles // 2)), tiles}):
        per = -(-tiles // ctas) if ctas else 1
        for stage_k in (0, 64, 256, 2048):
            for stages in (0, per + 1):
                out.append(dict(STREAM, clusters=ctas, stage_k=stage_k, stages=stages))
    return out


@pytest.mark.parametrize("case", FORCED, ids=_ids(FORCED))
def test_stream_every_variant(case):
    X, W = si.make_inputs(case)
    yref, A = reference(case, X, W)
    ran = 0
    for v in _variants(case):
        with sk.options(**v):
            b = Buffers(case, X, W, ldy=case.N + 7)
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
    assert ran >= len(_variants(case)) // 2


def test_stream_rows_do_not_depend_on_other_tokens():
    big = si.Case("st_rows16", M=16, N=384, K=8192, seed=1200)
    X, W = si.make_inputs(big)
    small = si.Case("st_rows11", M=11, N=384, K=8192, seed=1200)
    with sk.options(**STREAM, clusters=24, stages=3):
        b16 = Buffers(big, X, W)
        b11 = Buffers(small, X[:11].copy(), W)
        assert b16.run() == sk.SKINNY_OK and b11.run() == sk.SKINNY_OK
        y16, y11 = b16.y_mat(), b11.y_mat()
    assert np.array_equal(y16[:11].view(np.uint32), y11.view(np.uint32))


def test_stream_bf16_output_and_wrapper():
    case = si.Case("st_bf16", M=8, N=2112, K=7168, seed=1300, w_dist="uniform_isqrtk")
    X, W = si.make_inputs(case)
    yref, A = reference(case, X, W)
    x = torch.from_numpy(X.view(np.int16)).cuda().view(torch.bfloat16)
    w = torch.from_numpy(W.view(np.int16)).cuda().view(torch.bfloat16)
    with sk.options(**STREAM):
        y32 = sk.gemm(x, w)
        y16 = torch.empty(case.M, case.N, dtype=torch.bfloat16, device="cuda")
        sk.gemm(x, w, out=y16)
    torch.cuda.synchronize()
    check_parity(y32.cpu().numpy(), yref, A, case.name)
    assert torch.equal(y16.cpu(), y32.cpu().to(torch.bfloat16))


@pytest.mark.parametrize("pdl", [0, 1])
def test_stream_graph_chain_matches_eager(pdl):
    cases = [si.Case(f"st_g{i}", M=M, N=N, K=K, seed=1400 + i)
             for i, (M, N, K) in enumerate([(8, 2112, 7168), (2, 4096, 8192), (16, 1024, 4096)])]
    with sk.options(pdl=pdl, **STREAM):
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


def test_stream_timeout_path_reports_and_recovers():
    """A wait budget of 0 makes every bounded wait give up at once: the kernel
    records the error, drains the copies in flight and exits; the next call is
    exact."""
    case = si.Case("st_to", M=8, N=64, K=8192, seed=1500)
    X, W = si.make_inputs(case)
    assert sk.skinny_get_device_status() == 0
    with sk.options(wait_timeout_us=0, clusters=1, stages=6, **STREAM):
        b = Buffers(case, X, W)
        assert b.run() == sk.SKINNY_OK
        code = sk.skinny_get_device_status()
    assert code & 0xFF == sk.SKINNY_ERR_DEVICE_TIMEOUT
    assert (code >> 8) in (1, 2)
    assert sk.skinny_get_device_status() == 0
    with sk.options(clusters=1, stages=6, **STREAM):
        run_and_check(case)
    assert sk.skinny_get_device_status() == 0


def test_stream_misaligned_x_falls_back_when_not_forced():
    case = si.Case("st_xmis", M=4, N=7168, K=8192, seed=1600)
    b = run_and_check(case, x_offset=1)
    assert b.plan()["backend"] != sk.SKINNY_BACKEND_STREAM
