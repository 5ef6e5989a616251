"""GPU parity: the sm_103a kernels, called through the C ABI, against the oracle.

Bar (elementwise): |y - y_ref| <= 1e-5 * sum_k |x*w| + 1e-6, cosine >= 0.99999,
never a write outside Y[:M, :N], bit-identical results from run to run.
"""
import numpy as np
import pytest
import torch

import latency_skinny_bf16_gb300 as sk
import oracle
import skinny_inputs as si
from gpu_util import CANARY, Buffers, check_parity, reference, run_and_check

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True, scope="module")
def _init():
    assert sk.skinny_init(0) == sk.SKINNY_OK
    yield


def _ids(cases):
    return [c.name for c in cases]


# ---------------------------------------------------------------- the workloads, default dispatch

def rerun_same_bits(b):
    """Two more runs of the same call (PDL off, then mode 1), each into a
    freshly canaried Y: the bits of the first run, and nothing written
    outside Y[:M, :N]."""
    first = b.y_mat().copy()
    for pdl in (0, 1):
        b.y_dev.fill_(CANARY)
        with sk.options(pdl=pdl):
            assert b.run() == sk.SKINNY_OK
        assert np.array_equal(b.y_mat().view(np.uint32), first.view(np.uint32)), "run-to-run bits differ"
    assert b.canary_ok()


@pytest.mark.parametrize("case", si.router_small(), ids=_ids(si.router_small()))
def test_router_small(case):
    rerun_same_bits(run_and_check(case))


@pytest.mark.parametrize("case", si.dotprod_cases(), ids=_ids(si.dotprod_cases()))
def test_dotprod_regime(case):
    rerun_same_bits(run_and_check(case))


@pytest.mark.parametrize("case", si.splitk_cases(), ids=_ids(si.splitk_cases()))
def test_splitk_regime_and_bit_identity(case):
    X, W = si.make_inputs(case)
    b = Buffers(case, X, W)
    yref, A = reference(case, X, W)
    first = None
    for _ in range(10):
        assert b.run() == sk.SKINNY_OK
        y = b.y_mat().copy()
        if first is None:
            first = y
            check_parity(y, yref, A, case.name)
        else:
            assert np.array_equal(y.view(np.uint32), first.view(np.uint32)), "run-to-run bits differ"
    assert b.canary_ok()


@pytest.mark.parametrize("case", si.projection_cases(), ids=_ids(si.projection_cases()))
def test_projection_shapes_strided_output(case):
    """Parity against the oracle, then two more runs (the second with PDL in
    mode 1) that must give the same bits: the cluster reductions of these
    plans add their partials in a fixed order."""
    assert case.ly == case.N + 64
    rerun_same_bits(run_and_check(case))


EDGE = si.edge_cases()


@pytest.mark.parametrize("chunk", range(10))
def test_edge_cases(chunk):
    for case in EDGE[chunk * 20:(chunk + 1) * 20]:
        run_and_check(case)


# ---------------------------------------------------------------- every kernel variant, forced

FORCED_SHAPES = [
    si.Case("f_router", M=1, N=256, K=7168, seed=301),
    si.Case("f_ragged", M=3, N=37, K=2880, seed=302),          # N tail, K tail inside a chunk
    si.Case("f_m5", M=5, N=100, K=4096, seed=303),
    si.Case("f_m9", M=9, N=130, K=1040, seed=304),             # K % 256 != 0
    si.Case("f_m16", M=16, N=384, K=7168, seed=305),
    si.Case("f_k8", M=7, N=19, K=8, seed=306),                  # one vector of K
    si.Case("f_k16", M=16, N=17, K=16, seed=307),
    si.Case("f_bigk", M=2, N=48, K=14336, seed=308, w_dist="uniform_isqrtk"),
]


def _variants(case):
    out = []
    for bn in (1, 2, 4, 8):
        out.append(dict(backend=sk.SKINNY_BACKEND_DOTPROD, block_n=bn))
    if case.K % 32 == 0:
        for bn in (16, 32, 64):
            out.append(dict(backend=sk.SKINNY_BACKEND_DOTPROD, consumer=sk.SKINNY_CONSUMER_MMA, block_n=bn))
        if case.M <= 16:
            # K over a cluster of S CTAs (refused on the host when a rank would get no K)
            for s, bn in ((2, 16), (4, 64), (8, 16)):
                out.append(dict(backend=sk.SKINNY_BACKEND_DOTPROD, consumer=sk.SKINNY_CONSUMER_MMA, block_n=bn,
                                split_k=s))
    for cons in (sk.SKINNY_CONSUMER_FMA, sk.SKINNY_CONSUMER_MMA):
        if cons == sk.SKINNY_CONSUMER_MMA and case.K % 16:
            continue
        for s in (1, 2, 3, 8):
            for stages in (1, 2, 4):
                out.append(dict(backend=sk.SKINNY_BACKEND_SPLITK, consumer=cons, split_k=s, stages=stages))
    return out


@pytest.mark.parametrize("case", FORCED_SHAPES, ids=_ids(FORCED_SHAPES))
def test_every_variant(case):
    X, W = si.make_inputs(case)
    yref, A = reference(case, X, W)
    ran = 0
    for v in _variants(case):
        with sk.options(**v):
            b = Buffers(case, X, W, ldy=case.N + 3)
            st = b.run()
            if st == sk.SKINNY_ERR_UNSUPPORTED:
                # a forced plan that does not fit (e.g. the X slice of split_k=1
                # exceeds shared memory) is refused on the host, like the planner says
                with pytest.raises(sk.SkinnyError):
                    b.plan()
                continue
            assert st == sk.SKINNY_OK, (v, sk.skinny_status_string(st))
            check_parity(b.y_mat(), yref, A, f"{case.name} {v}")
            assert b.canary_ok(), v
            assert sk.skinny_get_device_status() == 0, v     # no bounded wait gave up
            ran += 1
    assert ran >= len(_variants(case)) // 2


@pytest.mark.parametrize("v", [dict(backend=1, block_n=2), dict(backend=1, consumer=2, block_n=16),
                               dict(backend=1, consumer=2, block_n=64)])
@pytest.mark.parametrize("M", [7, 16])
def test_small_x_chunks_in_dotprod(v, M):
    """K large enough that X is staged in several chunks."""
    case = si.Case("chunks", M=M, N=200, K=14336, seed=309, w_dist="uniform_isqrtk")
    with sk.options(**v):
        b = run_and_check(case, ldy=209)
        assert b.plan()["k_chunk"] < case.K
    assert sk.skinny_get_device_status() == 0


@pytest.mark.parametrize("M", [1, 3, 4, 8, 9, 16])
@pytest.mark.parametrize("bn", [16, 32, 64])
def test_dotmma_shapes(M, bn):
    """The tensor-core dot-product layout on ragged N, K = 32 * odd and strided X / Y."""
    case = si.Case("dm", M=M, N=16 * 9 + 7, K=32 * 45, seed=1000 + M)
    with sk.options(backend=sk.SKINNY_BACKEND_DOTPROD, consumer=sk.SKINNY_CONSUMER_MMA, block_n=bn):
        b = run_and_check(case, ldx=case.K + 40, ldy=case.N + 5)
        p = b.plan()
        assert (p["consumer"], p["block_n"]) == (sk.SKINNY_CONSUMER_MMA, bn)
        b2 = run_and_check(case, ldx=case.K + 3, x_offset=1)     # X rows not 16-byte aligned
    assert sk.skinny_get_device_status() == 0


@pytest.mark.parametrize("M", [1, 5, 9, 16])
@pytest.mark.parametrize("S,bn", [(2, 16), (3, 32), (4, 16), (8, 64)])
def test_dotmma_cluster_split(M, S, bn):
    """K cut over a cluster of S CTAs: ragged N, K = 32 * odd (a short last slice), X strided or
    misaligned (staged by plain loads), partials summed through DSMEM in rank order: bit-identical."""
    case = si.Case("dms", M=M, N=16 * 9 + 7, K=32 * 45, seed=1100 + 10 * M + S)
    with sk.options(backend=sk.SKINNY_BACKEND_DOTPROD, consumer=sk.SKINNY_CONSUMER_MMA, block_n=bn, split_k=S):
        b = run_and_check(case, ldx=case.K + 40, ldy=case.N + 5)
        p = b.plan()
        assert (p["consumer"], p["block_n"], p["split_k"]) == (sk.SKINNY_CONSUMER_MMA, bn, S)
        assert (p["grid_x"], p["grid_y"]) == (S, -(-case.N // bn))
        first = b.y_mat().copy()
        for _ in range(5):
            assert b.run() == sk.SKINNY_OK
            assert np.array_equal(b.y_mat().view(np.uint32), first.view(np.uint32))
        run_and_check(case, ldx=case.K + 3, x_offset=1)
    assert sk.skinny_get_device_status() == 0


@pytest.mark.parametrize("M,N,K,S", [(16, 256, 7168, 8), (12, 384, 7168, 4), (16, 256, 4096, 8), (8, 128, 2880, 2),
                                     (16, 2112, 7168, 2)])
def test_dotmma_cluster_split_router_shapes(M, N, K, S):
    """The router and projection shapes the cluster split serves, full size, against the oracle."""
    case = si.Case(f"dmr_M{M}_N{N}_K{K}_S{S}", M=M, N=N, K=K, seed=1200 + M + S, ldy=N + 64)
    with sk.options(backend=sk.SKINNY_BACKEND_DOTPROD, consumer=sk.SKINNY_CONSUMER_MMA, split_k=S):
        b = run_and_check(case)
        assert b.plan()["split_k"] == S
        assert b.canary_ok()
    assert sk.skinny_get_device_status() == 0


@pytest.mark.parametrize("M,N,K,S,bk,warps", [(5, 200, 14336, 2, 2048, 8), (16, 77, 7168, 4, 1024, 8),
                                              (9, 300, 7168, 2, 1024, 8), (16, 77, 7168, 4, 512, 4),
                                              (8, 150, 14336, 4, 1024, 8)])
def test_splitk_mma_consumer_warps(M, N, K, S, bk, warps):
    """The MMA consumer splits each stage over 8 warps when stages hold >= 1024 K elements
    (up to 16 tokens), else 4: both layouts against the oracle, bit-identical over runs."""
    case = si.Case(f"cw_M{M}_N{N}_K{K}_S{S}_bk{bk}", M=M, N=N, K=K, seed=1400 + M + S, ldy=N + 5)
    with sk.options(backend=sk.SKINNY_BACKEND_SPLITK, consumer=sk.SKINNY_CONSUMER_MMA, split_k=S, stage_k=bk):
        b = run_and_check(case)
        p = b.plan()
        assert (p["split_k"], p["stage_k"], p["threads"]) == (S, bk, (warps + 1) * 32), p
        first = b.y_mat().copy()
        for _ in range(3):
            assert b.run() == sk.SKINNY_OK
            assert np.array_equal(b.y_mat().view(np.uint32), first.view(np.uint32))
        assert b.canary_ok()
    assert sk.skinny_get_device_status() == 0


# ---------------------------------------------------------------- layouts: strides, offsets, alignment

@pytest.mark.parametrize("ldx_pad,ldw_pad,w_off,x_off", [
    (0, 0, 0, 0), (5, 0, 0, 0), (0, 3, 0, 0), (0, 8, 0, 0), (0, 0, 1, 0), (0, 0, 2, 0), (0, 0, 4, 0),
    (0, 1, 0, 1), (7, 5, 3, 3)])
@pytest.mark.parametrize("M", [1, 4, 8, 16])
def test_strides_and_misalignment(ldx_pad, ldw_pad, w_off, x_off, M):
    case = si.Case("lay", M=M, N=77, K=1000, seed=400 + M)
    b = run_and_check(case, ldx=case.K + ldx_pad, ldw=case.K + ldw_pad, ldy=case.N + 11,
                      w_offset=w_off, x_offset=x_off)
    p = b.plan()
    if w_off % 8 or (case.K + ldw_pad) % 8:
        assert p["backend"] == sk.SKINNY_BACKEND_DOTPROD and p["vec_elems"] < 8


def test_k_zero_writes_zeros_and_noop_sizes():
    case = si.Case("k0", M=3, N=10, K=0, seed=1)
    X = np.zeros((3, 0), np.uint16)
    W = np.zeros((10, 0), np.uint16)
    b = Buffers(case, X, W, ldx=1, ldw=1, ldy=13)
    assert b.run() == sk.SKINNY_OK
    assert np.all(b.y_mat() == 0.0) and b.canary_ok()
    y = torch.full((4,), 5.0, device="cuda")
    assert sk.skinny_gemm_bf16(0, 0, 0, 0, y.data_ptr(), 4, 0, 4, 8, 0) == sk.SKINNY_OK
    assert sk.skinny_gemm_bf16(0, 0, 0, 0, y.data_ptr(), 4, 2, 0, 8, 0) == sk.SKINNY_OK
    torch.cuda.synchronize()
    assert torch.all(y == 5.0)


def test_special_values():
    inf, nan, one, zero = 0x7F80, 0x7FC0, 0x3F80, 0x0000
    case = si.Case("sv", M=2, N=3, K=16, seed=0)
    X = np.full((2, 16), zero, np.uint16)
    W = np.full((3, 16), zero, np.uint16)
    X[0, 0], X[0, 1], X[1, 5] = inf, one, nan
    W[0, 0], W[0, 1], W[1, 1], W[2, 0], W[2, 3] = one, one, one, one, one
    yref, A = oracle.gemm(X, W, 2, 3, 16)
    for v in _variants(case):
        with sk.options(**v):
            b = Buffers(case, X, W)
            assert b.run() == sk.SKINNY_OK
            y = b.y_mat()
            assert np.array_equal(np.isnan(y), np.isnan(yref)), v
            assert np.array_equal(np.isinf(y), np.isinf(yref)), v


# ---------------------------------------------------------------- invariants on the GPU

@pytest.mark.parametrize("v", [dict(backend=1, block_n=1), dict(backend=1, block_n=4),
                               dict(backend=1, consumer=2, block_n=16), dict(backend=1, consumer=2, block_n=64),
                               dict(backend=2, consumer=1, split_k=8), dict(backend=2, consumer=2, split_k=4)])
def test_one_hot_rows_exact(v):
    K, N = 4096, 64
    case = si.Case("oh", M=1, N=N, K=K, seed=500)
    _, W = si.make_inputs(case)
    ks = [0, 1, 1000, 4095]
    X = np.zeros((len(ks), K), np.uint16)
    for i, k in enumerate(ks):
        X[i, k] = 0x3F80
    c = si.Case("oh", M=len(ks), N=N, K=K, seed=500)
    with sk.options(**v):
        b = Buffers(c, X, W)
        assert b.run() == sk.SKINNY_OK
        y = b.y_mat()
    for i, k in enumerate(ks):
        want = (W[:, k].astype(np.uint32) << 16).view(np.float32)
        assert np.array_equal(y[i], want)


@pytest.mark.parametrize("v", [dict(backend=1, block_n=2), dict(backend=1, consumer=2, block_n=32),
                               dict(backend=2, consumer=1, split_k=4), dict(backend=2, consumer=2, split_k=8)])
def test_row_independence_exact(v):
    case = si.Case("ri", M=8, N=96, K=7168, seed=501)
    X, W = si.make_inputs(case)
    with sk.options(**v):
        full = Buffers(case, X, W)
        assert full.run() == sk.SKINNY_OK
        yf = full.y_mat().copy()
        for m in range(8):
            one = Buffers(si.Case("ri1", M=1, N=96, K=7168, seed=501), X[m:m + 1], W)
            assert one.run() == sk.SKINNY_OK
            # each token's summation order does not depend on M under a fixed plan
            assert np.array_equal(one.y_mat()[0], yf[m]), m


def test_column_shards_match_full_call():
    """Output columns are independent: calling on row slices of W (shards of N)
    gives the full result; bit-exact under a plan that does not depend on N."""
    case = si.Case("shard", M=4, N=1024, K=7168, seed=502)
    X, W = si.make_inputs(case)
    with sk.options(backend=sk.SKINNY_BACKEND_DOTPROD, block_n=1):
        full = Buffers(case, X, W)
        assert full.run() == sk.SKINNY_OK
        yf = full.y_mat().copy()
        parts = []
        for n0, n1 in ((0, 256), (256, 640), (640, 1024)):
            c = si.Case("s", M=4, N=n1 - n0, K=7168, seed=0)
            b = Buffers(c, X, W[n0:n1])
            assert b.run() == sk.SKINNY_OK
            parts.append(b.y_mat().copy())
    assert np.array_equal(np.concatenate(parts, axis=1), yf)


# ---------------------------------------------------------------- PDL, graphs, the timeout path

def test_pdl_chain_on_off_bit_identical():
    case = si.pdl_chain_case()
    X, W = si.make_inputs(case)
    yref, A = reference(case, X, W)
    results = {}
    for pdl in (0, 1):
        with sk.options(pdl=pdl):
            bufs = [Buffers(case, X, W) for _ in range(4)]
            s = torch.cuda.current_stream().cuda_stream
            for i in range(64):
                assert bufs[i % 4].run(s) == sk.SKINNY_OK
            results[pdl] = [b.y_mat().copy() for b in bufs]
    for y0, y1 in zip(results[0], results[1]):
        assert np.array_equal(y0.view(np.uint32), y1.view(np.uint32))
        check_parity(y1, yref, A, "pdl chain")


@pytest.mark.parametrize("pdl", [0, 1])
def test_cuda_graph_capture_and_replay(pdl):
    cases = [si.Case("g1", M=2, N=256, K=7168, seed=601), si.Case("g2", M=12, N=384, K=7168, seed=602)]
    with sk.options(pdl=pdl):
        bufs, refs = [], []
        for c in cases:
            X, W = si.make_inputs(c)
            bufs.append(Buffers(c, X, W))
            refs.append(reference(c, X, W))
        s = torch.cuda.Stream()
        with torch.cuda.stream(s):
            for b in bufs:                       # eager once (also outside the capture)
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
        for b, e, (yref, A) in zip(bufs, eager, refs):
            assert np.array_equal(b.y_mat(), e)
            check_parity(b.y_mat(), yref, A, "graph")


@pytest.mark.parametrize("late", [0, 1])
def test_large_weight_graph_chain_with_pdl(late):
    """Calls on weights of 16 MB and more (the dot-product, split-K and tcgen05
    plans of the 30 and 75 MB projections), captured in one CUDA graph with PDL
    mode 1, the dependents' trigger at kernel entry (late = 0) or once each CTA
    has issued its last W load (late = 1): the replay gives the bits of the
    same calls run eagerly without PDL, within the parity bound."""
    cases = [si.Case(f"lw{i}", M=M, N=N, K=K, seed=6100 + i)
             for i, (M, N, K) in enumerate([(1, 2112, 7168), (8, 2112, 7168), (16, 2112, 7168),
                                            (3, 24576, 1536), (16, 24576, 1536)])]
    bufs = [Buffers(c, *si.make_inputs(c)) for c in cases]
    s = torch.cuda.Stream()
    with sk.options(pdl=0), torch.cuda.stream(s):
        for b in bufs:
            assert b.run(s.cuda_stream) == sk.SKINNY_OK
    torch.cuda.synchronize()
    eager = [b.y_mat().copy() for b in bufs]
    for b in bufs:
        b.y_dev.fill_(0.0)
    torch.cuda.synchronize()
    with sk.options(pdl=1, late_trigger=late):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            for b in bufs:
                assert b.run(s.cuda_stream) == sk.SKINNY_OK
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    assert sk.skinny_get_device_status() == 0
    for b, e, c in zip(bufs, eager, cases):
        assert np.array_equal(b.y_mat().view(np.uint32), e.view(np.uint32)), c.name
        X, W = si.make_inputs(c)
        yref, A = reference(c, X, W)
        check_parity(e, yref, A, c.name)


def test_timeout_path_reports_and_recovers():
    """A wait budget of 0 makes every bounded wait in the split-K kernel give
    up at once; the kernel records the error, drains its copies, takes part in
    the cluster barrier and exits.  Nothing hangs, and the next call is exact."""
    case = si.Case("to", M=8, N=64, K=7168, seed=700)
    X, W = si.make_inputs(case)
    assert sk.skinny_get_device_status() == 0
    with sk.options(backend=sk.SKINNY_BACKEND_SPLITK, consumer=sk.SKINNY_CONSUMER_FMA, split_k=2, stages=2,
                    wait_timeout_us=0):
        b = Buffers(case, X, W)
        assert b.run() == sk.SKINNY_OK
        code = sk.skinny_get_device_status()
    assert code & 0xFF == sk.SKINNY_ERR_DEVICE_TIMEOUT
    assert (code >> 8) in (1, 2, 4)
    assert sk.skinny_get_device_status() == 0          # read clears it
    with sk.options(backend=sk.SKINNY_BACKEND_SPLITK, consumer=sk.SKINNY_CONSUMER_FMA, split_k=2, stages=2):
        run_and_check(case)
    assert sk.skinny_get_device_status() == 0


@pytest.mark.parametrize("opts", [dict(backend=sk.SKINNY_BACKEND_DOTPROD, consumer=sk.SKINNY_CONSUMER_FMA),
                                  dict(backend=sk.SKINNY_BACKEND_DOTPROD, consumer=sk.SKINNY_CONSUMER_MMA),
                                  dict(backend=sk.SKINNY_BACKEND_DOTPROD, consumer=sk.SKINNY_CONSUMER_MMA,
                                       split_k=4, block_n=16)],
                         ids=["dotprod", "dotmma", "dotmma_split4"])
def test_dot_product_timeout_path_reports_and_recovers(opts):
    """The dot-product kernels' only wait is X staging by bulk copies: with a
    wait budget of 0 it gives up at once and is reported, the kernel still
    waits (bounded) for its copies before reading X, and the next call is
    exact."""
    case = si.Case("to_dot", M=8, N=256, K=4096, seed=701)
    X, W = si.make_inputs(case)
    assert sk.skinny_get_device_status() == 0
    with sk.options(wait_timeout_us=0, **opts):
        b = Buffers(case, X, W)
        assert b.run() == sk.SKINNY_OK
        code = sk.skinny_get_device_status()
    assert code & 0xFF == sk.SKINNY_ERR_DEVICE_TIMEOUT
    assert (code >> 8) == 4                # the X-staging wait
    assert sk.skinny_get_device_status() == 0
    with sk.options(**opts):
        run_and_check(case)
    assert sk.skinny_get_device_status() == 0


def test_tensor_wrapper():
    case = si.Case("tw", M=5, N=300, K=2048, seed=800)
    X, W = si.make_inputs(case)
    x = torch.from_numpy(X.view(np.int16)).cuda().view(torch.bfloat16)
    w = torch.from_numpy(W.view(np.int16)).cuda().view(torch.bfloat16)
    out = torch.full((5, 320), -1.0, device="cuda")[:, :300]
    sk.gemm(x, w, out=out)
    torch.cuda.synchronize()
    yref, A = reference(case, X, W)
    check_parity(out.cpu().numpy(), yref, A, "wrapper")
    with pytest.raises(TypeError):
        sk.gemm(x.float(), w)
    with pytest.raises(sk.SkinnyError):
        sk.gemm(torch.zeros(65, 2048, dtype=torch.bfloat16, device="cuda"), w)   # M > 64


PERSISTENT_CFGS = [  # (split_k, clusters, stages, stage_k)
    (1, 3, 2, 0), (1, 7, 8, 256), (2, 5, 4, 0), (4, 2, 3, 0), (8, 3, 2, 0), (8, 2, 16, 0), (4, 3, 16, 0),
    (1, 2, 10, 256), (1, 3, 2, 1024), (2, 5, 3, 512), (8, 2, 2, 64), (2, 4, 2, 2048), (4, 3, 5, 192)]


def persistent_case(cons, split):
    return si.Case("pers", M=11 if cons == sk.SKINNY_CONSUMER_MMA else 6, N=16 * 13 + 5, K=4096, seed=900 + split)


@pytest.mark.parametrize("cons", [sk.SKINNY_CONSUMER_FMA, sk.SKINNY_CONSUMER_MMA])
@pytest.mark.parametrize("split,clusters,stages,stage_k", PERSISTENT_CFGS)
def test_persistent_clusters(cons, split, clusters, stages, stage_k):
    """Clusters that loop over several 16-row tiles (tile = y, y + C, ...): the
    ring streams across tile boundaries and the DSMEM slots alternate between
    two buffers, one cluster-barrier phase per tile."""
    case = persistent_case(cons, split)
    X, W = si.make_inputs(case)
    yref, A = reference(case, X, W)
    with sk.options(backend=sk.SKINNY_BACKEND_SPLITK, consumer=cons, split_k=split, clusters=clusters,
                    stages=stages, stage_k=stage_k):
        b = Buffers(case, X, W, ldy=case.N + 9)
        try:
            p = b.plan()
        except sk.SkinnyError as e:      # a forced plan that does not fit shared memory
            assert e.status == sk.SKINNY_ERR_UNSUPPORTED and b.run() == sk.SKINNY_ERR_UNSUPPORTED
            pytest.skip("forced plan does not fit shared memory")
        assert (p["grid_x"], p["grid_y"]) == (split, clusters)
        if stage_k:
            assert p["stage_k"] == stage_k
        first = None
        for _ in range(3):
            assert b.run() == sk.SKINNY_OK
            y = b.y_mat().copy()
            if first is None:
                first = y
                check_parity(y, yref, A, f"persistent S={split} C={clusters}")
            else:
                assert np.array_equal(y.view(np.uint32), first.view(np.uint32))
        assert b.canary_ok()
    assert sk.skinny_get_device_status() == 0


# ---------------------------------------------------------------- bf16 output

def _bf16_round(y32: np.ndarray) -> np.ndarray:
    """fp32 -> bf16 round-to-nearest-even by PyTorch's conversion, as bit patterns."""
    return torch.from_numpy(np.ascontiguousarray(y32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


BF16_SHAPES = [si.Case("b_router", M=4, N=256, K=7168, seed=1101),
               si.Case("b_ragged", M=9, N=37, K=2880, seed=1102),
               si.Case("b_odd", M=3, N=50, K=1001, seed=1103, x_dist="normal", w_dist="normal", outliers=True)]


@pytest.mark.parametrize("case", BF16_SHAPES, ids=_ids(BF16_SHAPES))
def test_bf16_output_every_variant(case):
    """bf16 Y is the fp32 result of the same plan rounded once to nearest-even:
    bit-exact against the fp32 entry point's output rounded by PyTorch, and
    within the fp32 bound plus one bf16 ulp of the oracle.  Gaps untouched."""
    X, W = si.make_inputs(case)
    yref, A = reference(case, X, W)
    ldy = case.N + 5
    for v in _variants(case):
        with sk.options(**v):
            b = Buffers(case, X, W, ldy=ldy)
            st = b.run()
            if st == sk.SKINNY_ERR_UNSUPPORTED:
                continue
            assert st == sk.SKINNY_OK
            y32 = b.y_mat().copy()
            yb = torch.full((case.M * ldy + 16,), 0x7FC1, dtype=torch.int16, device="cuda")   # canary: a NaN pattern
            st = sk.skinny_gemm_bf16_bf16out(b.x_ptr, b.ldx, b.w_ptr, b.ldw, yb.data_ptr(), ldy, case.M, case.N,
                                             case.K, 0)
            assert st == sk.SKINNY_OK, v
            torch.cuda.synchronize()
            ybits = yb.cpu().numpy().view(np.uint16)
            body = ybits[: case.M * ldy].reshape(case.M, ldy)
            assert np.array_equal(body[:, : case.N], _bf16_round(y32)), v
            assert np.all(body[:, case.N:] == 0x7FC1) and np.all(ybits[case.M * ldy:] == 0x7FC1), v
            yv = (body[:, : case.N].astype(np.uint32) << 16).view(np.float32).astype(np.float64)
            fin = np.isfinite(yref)
            err = np.abs(yv[fin] - yref[fin])
            assert np.all(err <= 1e-5 * A[fin] + 1e-6 + 2.0 ** -8 * np.abs(yref[fin])), v
    assert sk.skinny_get_device_status() == 0


def test_bf16_output_k_zero_and_wrapper():
    yb = torch.full((3, 9), 7.0, dtype=torch.bfloat16, device="cuda")
    assert sk.skinny_gemm_bf16_bf16out(0, 0, 0, 0, yb.data_ptr(), 9, 3, 8, 0, 0) == sk.SKINNY_OK
    torch.cuda.synchronize()
    assert torch.all(yb[:, :8] == 0) and torch.all(yb[:, 8] == 7.0)
    case = si.Case("bw", M=6, N=300, K=2048, seed=1104)
    X, W = si.make_inputs(case)
    x = torch.from_numpy(X.view(np.int16)).cuda().view(torch.bfloat16)
    w = torch.from_numpy(W.view(np.int16)).cuda().view(torch.bfloat16)
    out32 = sk.gemm(x, w)
    out16 = sk.gemm(x, w, out=torch.empty(6, 300, dtype=torch.bfloat16, device="cuda"))
    torch.cuda.synchronize()
    assert torch.equal(out16, out32.to(torch.bfloat16))
