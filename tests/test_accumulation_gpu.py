"""Long-K accumulation on same-sign operands, every backend, against the oracle.

Random-sign inputs let the rounding errors of a long fp32 sum cancel; here
every product x*w is positive (X ~ |N(0,1)|, W ~ |N(0,1)| or U(0, 1/sqrt(K))),
so nothing cancels and a biased rounding (for example a tensor core that
truncates inside its accumulation) grows linearly with the chain length.  K
reaches 14336 (the longest projection), so a tcgen05 accumulator without a
K split chains 896 MMAs of K = 16 per output.

The bar is the one every other parity test uses: |y - y_ref| <= 1e-5 *
sum_k |x*w| + 1e-6 elementwise (here sum_k |x*w| = y_ref), cosine >=
0.99999.  Each case also prints the largest err / A it saw, a record of the
margin per backend.
"""
import numpy as np
import pytest

import latency_skinny_bf16_gb300 as sk
import skinny_inputs as si
from gpu_util import Buffers, check_parity, reference

pytestmark = pytest.mark.gpu

TC = sk.SKINNY_BACKEND_TCGEN05
DOT = sk.SKINNY_BACKEND_DOTPROD
SPLIT = sk.SKINNY_BACKEND_SPLITK
STREAM = sk.SKINNY_BACKEND_STREAM
MMA = sk.SKINNY_CONSUMER_MMA
FMA = sk.SKINNY_CONSUMER_FMA


@pytest.fixture(autouse=True, scope="module")
def _init():
    assert sk.skinny_init(0) == sk.SKINNY_OK
    yield


# (name, forced options, token counts it takes)
VARIANTS = [
    ("tc_s1_bn128", dict(backend=TC, split_k=1, block_n=128, stage_k=128), (1, 8, 16, 32, 64)),
    ("tc_s1_bn64", dict(backend=TC, split_k=1, block_n=64, stage_k=128), (1, 16, 64)),
    ("tc_s4_bn128", dict(backend=TC, split_k=4, block_n=128, stage_k=128), (8, 16, 64)),
    ("tc_tuned", dict(backend=TC), (2, 16, 40)),
    ("dotmma", dict(backend=DOT, consumer=MMA), (4, 8, 16, 32, 64)),
    ("dotmma_s4", dict(backend=DOT, consumer=MMA, split_k=4), (4, 16)),
    ("splitk_mma_s4", dict(backend=SPLIT, consumer=MMA, split_k=4), (5, 16, 32)),
    ("splitk_mma_s8", dict(backend=SPLIT, consumer=MMA, split_k=8), (8, 16, 64)),
    ("splitk_fma_s8", dict(backend=SPLIT, consumer=FMA, split_k=8), (5, 16)),
    ("stream", dict(backend=STREAM), (4, 16)),
    ("dotprod_fma", dict(backend=DOT, consumer=FMA), (1, 4, 16)),
]

SHAPES = [
    # (N, K, x_dist, w_dist)
    (256, 14336, "abs_normal", "abs_normal"),
    (300, 14336, "abs_normal", "abs_uniform_isqrtk"),
    (192, 7168, "abs_normal", "abs_normal"),
]

CASES = []
for vname, opts, tokens in VARIANTS:
    for si_, (N, K, xd, wd) in enumerate(SHAPES):
        for M in tokens:
            CASES.append((vname, opts, si.Case(f"acc_{vname}_M{M}_N{N}_K{K}_{wd}", M=M, N=N, K=K,
                                               seed=7000 + 101 * si_ + M, x_dist=xd, w_dist=wd, ldy=N + 4)))


@pytest.mark.parametrize("vname,opts,case", CASES, ids=[c.name for _, _, c in CASES])
def test_same_sign_long_k(vname, opts, case):
    X, W = si.make_inputs(case)
    with sk.options(**opts):
        b = Buffers(case, X, W)
        try:
            p = b.plan()
        except sk.SkinnyError as e:
            if e.status != sk.SKINNY_ERR_UNSUPPORTED:
                raise
            assert b.run() == sk.SKINNY_ERR_UNSUPPORTED        # refused on the host, as planned
            pytest.skip(f"{vname}: no plan for M={case.M} K={case.K} (refused on the host)")
        if "backend" in opts:
            assert p["backend"] == opts["backend"], (vname, p)
        assert b.run() == sk.SKINNY_OK
        y = b.y_mat().copy()
    yref, A = reference(case, X, W)
    assert np.all(A > 0) and np.allclose(A, yref)       # every product is positive
    worst = check_parity(y, yref, A, case.name)
    signed = float(np.max(np.abs(y.astype(np.float64) - yref) / A))
    bias = float(np.mean((y.astype(np.float64) - yref) / A))
    print(f"ACCUM {vname} M={case.M} N={case.N} K={case.K} w={case.w_dist} split_k={p['split_k']} "
          f"max_err_over_A={worst:.3e} mean_signed_err_over_A={bias:+.3e}")
    assert signed <= 1e-5
    assert b.canary_ok()
    assert sk.skinny_get_device_status() == 0
