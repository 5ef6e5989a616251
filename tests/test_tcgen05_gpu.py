"""GPU parity of the tcgen05 backend (128 W rows per CTA on the fifth-generation
tensor cores, accumulator in tensor memory, W / X boxes by tensor-map TMA,
optional cluster split-K) against the oracle, through the C ABI.

Same bar as the other backends: |y - y_ref| <= 1e-5 * sum_k |x*w| + 1e-6
elementwise, cosine >= 0.99999, nothing written outside Y[:M, :N], and
bit-identical results from run to run under one plan.
"""
import numpy as np
import pytest
import torch

import latency_skinny_bf16_gb300 as sk
import oracle
import skinny_inputs as si
from gpu_util import Buffers, check_parity, reference, run_and_check
from plan_checks import check_tc_geometry

pytestmark = pytest.mark.gpu

TC = dict(backend=sk.SKINNY_BACKEND_TCGEN05)


@pytest.fixture(autouse=True, scope="module")
def _init():
    assert sk.skinny_init(0) == sk.SKINNY_OK
    yield


def _ids(cases):
    return [c.name for c in cases]


def _run_twice(b, yref, A, what):
    first = None
    for _ in range(2):
        assert b.run() == sk.SKINNY_OK, what
        y = b.y_mat().copy()
        if first is None:
            first = y
            check_parity(y, yref, A, what)
        else:
            assert np.array_equal(y.view(np.uint32), first.view(np.uint32)), f"{what}: run-to-run bits differ"
    assert b.canary_ok(), f"{what}: wrote outside Y[:M, :N]"


# every token bucket (16 / 32 / 64 MMA columns, with rows past M), ragged N
# (partial 128-row tiles), K tails that are not a multiple of the 64-element box
SHAPES = [(130, 1536), (300, 576), (64, 4104), (1000, 2048)]
TOKENS = [1, 3, 8, 16, 17, 31, 32, 33, 50, 64]
CASES = [si.Case(f"tc_M{M}_N{N}_K{K}", M=M, N=N, K=K, seed=5000 + 37 * i + M, w_dist="uniform_isqrtk", ldy=N + 3)
         for i, (N, K) in enumerate(SHAPES) for M in TOKENS]


@pytest.mark.parametrize("bn", [128, 64])
@pytest.mark.parametrize("case", CASES, ids=_ids(CASES))
def test_tc_default_plan(case, bn):
    X, W = si.make_inputs(case)
    with sk.options(block_n=bn, **TC):
        b = Buffers(case, X, W)
        p = b.plan()
        assert (p["backend"], p["block_n"]) == (sk.SKINNY_BACKEND_TCGEN05, bn)
        check_tc_geometry(p, case.M, case.N, case.K)
        yref, A = reference(case, X, W)
        _run_twice(b, yref, A, case.name)
    assert sk.skinny_get_device_status() == 0


VARIANT_CASES = [
    si.Case("tcv_m5", M=5, N=200, K=1000, seed=5101),                        # K % 64 != 0
    si.Case("tcv_m40", M=40, N=129, K=2048, seed=5102, outliers=True),       # one row past a tile
    si.Case("tcv_m64", M=64, N=256, K=520, seed=5103, w_dist="normal"),
    si.Case("tcv_k8", M=16, N=128, K=8, seed=5104),                          # one box, mostly zero fill
    si.Case("tcv_n1", M=1, N=1, K=64, seed=5105),
    si.Case("tcv_k200", M=24, N=77, K=200, seed=5106),                       # S = 8 leaves ranks empty
]


def _variants():
    out = []
    for bn in (128, 64):
        for s in (1, 2, 4, 8):
            for stages in (1, 2, 3, 6):
                for stage_k in (64, 128, 256):
                    out.append(dict(block_n=bn, split_k=s, stages=stages, stage_k=stage_k, **TC))
    return out


@pytest.mark.parametrize("case", VARIANT_CASES, ids=_ids(VARIANT_CASES))
def test_tc_every_variant(case):
    """Cluster sizes 1..8 (empty K slices included), ring depths down to one
    stage (the producer waits on every stage), 1..4 boxes per stage."""
    X, W = si.make_inputs(case)
    yref, A = reference(case, X, W)
    ran = 0
    for v in _variants():
        with sk.options(**v):
            b = Buffers(case, X, W, ldy=case.N + 5)
            st = b.run()
            if st == sk.SKINNY_ERR_UNSUPPORTED:
                with pytest.raises(sk.SkinnyError):   # refused on the host, as the planner says
                    b.plan()
                continue
            assert st == sk.SKINNY_OK, (v, sk.skinny_status_string(st))
            p = b.plan()
            assert (p["block_n"], p["split_k"], p["stages"], p["stage_k"]) == \
                (v["block_n"], v["split_k"], v["stages"], v["stage_k"])
            check_parity(b.y_mat(), yref, A, f"{case.name} {v}")
            assert b.canary_ok(), v
            assert sk.skinny_get_device_status() == 0, v
            ran += 1
    # refused: rings beyond shared memory, and split rings too small for the partials
    assert ran >= len(_variants()) // 2


@pytest.mark.parametrize("ldx_pad,ldw_pad,w_off", [(8, 0, 0), (0, 16, 0), (0, 0, 8), (24, 8, 64)])
@pytest.mark.parametrize("M", [2, 16, 48])
def test_tc_strides(ldx_pad, ldw_pad, w_off, M):
    """Padded rows and a shifted (still 16-byte aligned) W base."""
    case = si.Case(f"tc_ld_{M}_{ldx_pad}_{ldw_pad}_{w_off}", M=M, N=333, K=1536, seed=5200 + M + ldx_pad + w_off)
    with sk.options(**TC):
        b = run_and_check(case, ldx=case.K + ldx_pad, ldw=case.K + ldw_pad, ldy=case.N + 1, w_offset=w_off)
        assert b.plan()["backend"] == sk.SKINNY_BACKEND_TCGEN05
    assert sk.skinny_get_device_status() == 0


@pytest.mark.parametrize("ldx_pad,x_off,w_off", [(3, 0, 0), (0, 1, 0), (0, 0, 4)])
def test_tc_needs_16_byte_rows(ldx_pad, x_off, w_off):
    """Rows that are not 16-byte aligned are refused on the host when the
    backend is forced, and take another backend when it is not."""
    case = si.Case(f"tc_mis_{ldx_pad}_{x_off}_{w_off}", M=12, N=256, K=1024, seed=5300 + ldx_pad + x_off + w_off)
    X, W = si.make_inputs(case)
    with sk.options(**TC):
        b = Buffers(case, X, W, ldx=case.K + ldx_pad, x_offset=x_off, w_offset=w_off)
        assert b.run() == sk.SKINNY_ERR_UNSUPPORTED
    b = run_and_check(case, ldx=case.K + ldx_pad, x_offset=x_off, w_offset=w_off)
    assert b.plan()["backend"] != sk.SKINNY_BACKEND_TCGEN05


@pytest.mark.parametrize("bn", [128, 64])
@pytest.mark.parametrize("M", [1, 16, 64])
@pytest.mark.parametrize("N,K", [(24576, 1536), (7168, 14336), (2112, 7168)])
def test_tc_projection_shapes_sampled(M, N, K, bn):
    """The decode projection weights at full size, in the default tcgen05 plan
    for them at each tile height; 512 output columns checked against the oracle."""
    case = si.Case(f"tc_proj_M{M}_{N}x{K}", M=M, N=N, K=K, seed=5400 + M + N % 97, w_dist="uniform_isqrtk")
    X, W = si.make_inputs(case)
    with sk.options(block_n=bn, **TC):
        b = Buffers(case, X, W)
        first = None
        for _ in range(2):
            assert b.run() == sk.SKINNY_OK
            y = b.y_mat().copy()
            if first is None:
                first = y
            else:
                assert np.array_equal(y.view(np.uint32), first.view(np.uint32))
        assert b.canary_ok()
    cols = np.sort(np.random.default_rng(case.seed).choice(N, 512, replace=False))
    cols[-1] = N - 1                                    # the last (ragged-free) tile's last row
    yref, A = oracle.gemm(X, np.ascontiguousarray(W[cols]), M, len(cols), K)
    check_parity(first[:, cols], yref, A, case.name)
    assert sk.skinny_get_device_status() == 0


def test_tc_rows_do_not_depend_on_other_tokens():
    """Within one token bucket and one plan, the first rows of a 64-token call
    equal a 40-token call on the same rows bit for bit."""
    big = si.Case("tc_rows64", M=64, N=384, K=4096, seed=5500)
    X, W = si.make_inputs(big)
    small = si.Case("tc_rows40", M=40, N=384, K=4096, seed=5500)
    for s, bn in ((1, 128), (4, 128), (2, 64)):
        with sk.options(split_k=s, stages=4, block_n=bn, **TC):
            b64 = Buffers(big, X, W)
            b40 = Buffers(small, X[:40].copy(), W)
            assert b64.run() == sk.SKINNY_OK and b40.run() == sk.SKINNY_OK
            y64, y40 = b64.y_mat(), b40.y_mat()
        assert np.array_equal(y64[:40].view(np.uint32), y40.view(np.uint32)), s


def test_tc_bf16_output():
    case = si.Case("tc_bf16", M=24, N=2112, K=7168, seed=5600, w_dist="uniform_isqrtk")
    X, W = si.make_inputs(case)
    yref, A = reference(case, X, W)
    x = torch.from_numpy(X.view(np.int16)).cuda().view(torch.bfloat16)
    w = torch.from_numpy(W.view(np.int16)).cuda().view(torch.bfloat16)
    with sk.options(**TC):
        y32 = sk.gemm(x, w)
        y16 = torch.empty(case.M, case.N, dtype=torch.bfloat16, device="cuda")
        sk.gemm(x, w, out=y16)
        torch.cuda.synchronize()
    check_parity(y32.cpu().numpy(), yref, A, case.name)
    assert torch.equal(y16.cpu(), y32.cpu().to(torch.bfloat16))


@pytest.mark.parametrize("pdl", [0, 1])
def test_tc_graph_capture_chain(pdl):
    """A chain of calls captured in a CUDA graph, with and without PDL, writing
    one Y after another: the replay reproduces the eager results bit for bit."""
    cases = [si.Case(f"tc_g{i}", M=M, N=N, K=K, seed=5700 + i)
             for i, (M, N, K) in enumerate([(17, 256, 7168), (64, 384, 4096), (8, 2112, 7168), (32, 1000, 1536)])]
    with sk.options(pdl=pdl, **TC):
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
        X, W = si.make_inputs(c)
        yref, A = reference(c, X, W)
        check_parity(e, yref, A, c.name)
    assert sk.skinny_get_device_status() == 0


@pytest.mark.parametrize("split_k,bn", [(1, 128), (4, 128), (2, 64)])
def test_tc_timeout_path_reports_and_recovers(split_k, bn):
    """A wait budget of 0 makes every bounded wait give up at once: the kernel
    records the error, drains the copies in flight, takes part in both cluster
    barriers, frees its tensor memory and exits; the next call is exact."""
    case = si.Case(f"tc_to{split_k}", M=16, N=256, K=8192, seed=5800 + split_k)
    X, W = si.make_inputs(case)
    assert sk.skinny_get_device_status() == 0
    with sk.options(wait_timeout_us=0, split_k=split_k, stages=4, block_n=bn, **TC):
        b = Buffers(case, X, W)
        assert b.run() == sk.SKINNY_OK
        code = sk.skinny_get_device_status()
    assert code & 0xFF == sk.SKINNY_ERR_DEVICE_TIMEOUT
    assert (code >> 8) in (1, 2, 5, 6)
    assert sk.skinny_get_device_status() == 0
    with sk.options(split_k=split_k, stages=4, block_n=bn, **TC):
        run_and_check(case)
    assert sk.skinny_get_device_status() == 0


@pytest.mark.parametrize("M,N,K", [(20, 300, 1000), (17, 64, 4104), (64, 256, 14336)])
def test_tc_takes_medium_m_shapes_the_other_backends_cannot(M, N, K):
    """Unforced: 17..64 tokens with K % 16 != 0, or 64 tokens whose split-K X
    slice does not fit shared memory, run on tcgen05 (16-byte aligned rows)."""
    case = si.Case(f"tc_route_M{M}_N{N}_K{K}", M=M, N=N, K=K, seed=5900 + M + K % 97, w_dist="uniform_isqrtk",
                   ldy=N + 2)
    b = run_and_check(case)
    assert b.plan()["backend"] == sk.SKINNY_BACKEND_TCGEN05
    assert sk.skinny_get_device_status() == 0
