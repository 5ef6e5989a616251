"""Host-side tests of the C ABI: no GPU needed, no kernel launched.

The library must load and export every function that ``include/*.h``
declares; every argument error must be reported on the host before any CUDA
call; the dispatcher (``skinny_plan_for``) is a pure function of the shapes,
pointers and the SM count.
"""
import glob
import os
import re

import pytest

import latency_skinny_bf16_gb300 as sk
from plan_checks import check_tc_geometry

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
A16 = 0x7F0000000000        # fake, 16-byte aligned "device" addresses: never dereferenced
B16 = 0x7F0010000000
C16 = 0x7F0020000000


def declared_functions():
    names = []
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        with open(h) as f:
            src = f.read()
        names += re.findall(r"SKINNY_API\s+[\w\s\*]+?\b(\w+)\s*\(", src)
    return names


def test_library_exports_every_declared_symbol():
    lib = sk.load_library()
    names = declared_functions()
    assert len(names) >= 9
    for n in names:
        assert hasattr(lib, n), f"{n} declared in include/ but not exported"
    assert set(sk.EXPORTED_SYMBOLS) <= set(names)
    assert sk.skinny_version() >= 100


def test_status_strings():
    for code in range(7):
        assert sk.skinny_status_string(code).startswith("SKINNY_")
    assert sk.skinny_status_string(99) == "SKINNY_ERR_UNKNOWN"


def call(X=A16, ldx=64, W=B16, ldw=64, Y=C16, ldy=32, M=4, N=32, K=64):
    return sk.skinny_gemm_bf16(X, ldx, W, ldw, Y, ldy, M, N, K, 0)


@pytest.mark.parametrize("kw,expect", [
    (dict(M=-1), sk.SKINNY_ERR_INVALID_VALUE),
    (dict(N=-1), sk.SKINNY_ERR_INVALID_VALUE),
    (dict(K=-1), sk.SKINNY_ERR_INVALID_VALUE),
    (dict(M=65), sk.SKINNY_ERR_UNSUPPORTED),
    (dict(M=1000), sk.SKINNY_ERR_UNSUPPORTED),
    (dict(M=0), sk.SKINNY_OK),
    (dict(N=0), sk.SKINNY_OK),
    (dict(M=0, X=0, W=0, Y=0), sk.SKINNY_OK),
    (dict(ldx=63), sk.SKINNY_ERR_INVALID_VALUE),
    (dict(ldw=10), sk.SKINNY_ERR_INVALID_VALUE),
    (dict(ldy=31), sk.SKINNY_ERR_INVALID_VALUE),
    (dict(X=0), sk.SKINNY_ERR_INVALID_VALUE),
    (dict(W=0), sk.SKINNY_ERR_INVALID_VALUE),
    (dict(Y=0), sk.SKINNY_ERR_INVALID_VALUE),
    (dict(X=A16 + 1), sk.SKINNY_ERR_MISALIGNED),
    (dict(W=B16 + 3), sk.SKINNY_ERR_MISALIGNED),
    (dict(Y=C16 + 2), sk.SKINNY_ERR_MISALIGNED),
    (dict(Y=A16 + 64), sk.SKINNY_ERR_INVALID_VALUE),      # Y overlaps X
    (dict(Y=B16 + 2048), sk.SKINNY_ERR_INVALID_VALUE),    # Y overlaps W
])
def test_argument_errors_are_host_side(kw, expect):
    assert call(**kw) == expect


def test_k_zero_needs_only_y():
    # K == 0: X and W are not read, so NULL is allowed; Y must still be valid
    assert sk.skinny_plan_for(0, 0, 0, 0, C16, 32, 4, 32, 0, 152)["backend"] == 0
    with pytest.raises(sk.SkinnyError):
        sk.skinny_plan_for(0, 0, 0, 0, 0, 32, 4, 32, 0, 152)


@pytest.mark.skipif(__import__("torch").cuda.is_available(), reason="checks the no-device answer")
def test_valid_call_without_device_reports_no_device():
    assert call() == sk.SKINNY_ERR_NO_DEVICE
    assert sk.skinny_init(0) == sk.SKINNY_ERR_NO_DEVICE


def plan(M, N, K, ldw=None, W=B16, num_sms=152, X=A16, ldx=None, Y=C16, ldy=None):
    return sk.skinny_plan_for(X, ldx or K, W, ldw or K, Y, ldy or N, M, N, K, num_sms)


# shapes below are not in the tuning table, so they exercise the default rule
def test_default_rule_dotprod_small_m_or_short_k():
    for M in (1, 2, 3, 4):
        assert plan(M, 320, 7168)["backend"] == sk.SKINNY_BACKEND_DOTPROD
        assert plan(M, 320, 7168)["tuned"] == 0
    assert plan(8, 256, 1024)["backend"] == sk.SKINNY_BACKEND_DOTPROD   # K < 2048


def test_default_rule_splitk_larger_m():
    for M in (5, 8, 12, 16):
        p = plan(M, 256, 7200)
        assert p["backend"] == sk.SKINNY_BACKEND_SPLITK
        assert 1 <= p["split_k"] <= 8 and p["grid_x"] == p["split_k"]
        assert p["grid_y"] == 16 and p["block_n"] == 16
        assert p["smem_bytes"] <= 227 * 1024
        assert p["split_k"] * p["k_chunk"] >= 7200 and p["k_chunk"] % 16 == 0


def test_vector_width_follows_alignment():
    assert plan(1, 256, 7168)["vec_elems"] == 8
    assert plan(1, 256, 7168, W=B16 + 8)["vec_elems"] == 4
    assert plan(1, 256, 7168, W=B16 + 4)["vec_elems"] == 2
    assert plan(1, 256, 7168, W=B16 + 2)["vec_elems"] == 1
    assert plan(1, 256, 7170)["vec_elems"] == 2       # ldw = K = 7170: rows 4-byte aligned
    assert plan(1, 256, 7169)["vec_elems"] == 1       # odd ldw: rows 2-byte aligned
    assert plan(1, 256, 2884)["vec_elems"] == 4


def test_misaligned_weights_never_take_splitk():
    for W, K in ((B16 + 2, 7168), (B16, 7169), (B16, 7172)):
        assert plan(16, 256, K, W=W)["backend"] == sk.SKINNY_BACKEND_DOTPROD


def test_dotprod_block_n_grows_with_n():
    assert plan(1, 256, 7200)["block_n"] == 1
    assert plan(1, 24576, 1504)["block_n"] == 8


def test_default_rule_tensor_core_dotprod_for_large_weights():
    p = plan(8, 8192, 3072)          # 48 MB of W, not tuned, K < 4096 (longer K streams)
    assert (p["backend"], p["consumer"]) == (sk.SKINNY_BACKEND_DOTPROD, sk.SKINNY_CONSUMER_MMA)
    assert p["block_n"] in (16, 32, 64) and p["grid_x"] * p["block_n"] >= 8192
    p = plan(2, 2112, 7168)
    blocks = p["grid_y"] if p["split_k"] > 1 else p["grid_x"]     # a cluster split: grid split_k x blocks
    assert blocks * p["block_n"] >= 2112


def test_x_chunking_for_large_m_times_k():
    p = plan(16, 7168, 14336, ldy=7168 + 64)
    if p["backend"] == sk.SKINNY_BACKEND_DOTPROD:
        assert p["k_chunk"] < 14336
    else:
        assert p["split_k"] * p["k_chunk"] >= 14336
    assert p["smem_bytes"] <= 227 * 1024


def test_forced_options_and_restore():
    with sk.options(backend=sk.SKINNY_BACKEND_SPLITK, consumer=sk.SKINNY_CONSUMER_FMA, split_k=4, stages=2):
        p = plan(3, 256, 7168)
        assert (p["backend"], p["consumer"], p["split_k"], p["stages"]) == (2, 1, 4, 2)
        with pytest.raises(sk.SkinnyError):      # split-K cannot read misaligned W rows
            plan(3, 256, 7169)
    with sk.options(backend=sk.SKINNY_BACKEND_DOTPROD, block_n=4):
        p = plan(16, 256, 7168)
        assert (p["backend"], p["block_n"]) == (1, 4)
    assert sk.skinny_get_option(sk.SKINNY_OPT_FORCE_BACKEND) == 0
    assert sk.skinny_get_option(sk.SKINNY_OPT_FORCE_BLOCK_N) == 0
    with sk.options(backend=sk.SKINNY_BACKEND_SPLITK, consumer=sk.SKINNY_CONSUMER_MMA):
        with pytest.raises(sk.SkinnyError):      # MMA needs K % 16 == 0
            plan(8, 256, 7176)


@pytest.mark.parametrize("opt,bad", [(sk.SKINNY_OPT_PDL, 3), (sk.SKINNY_OPT_FORCE_BACKEND, 5),
                                     (sk.SKINNY_OPT_FORCE_SPLIT_K, 9), (sk.SKINNY_OPT_FORCE_BLOCK_N, 3),
                                     (sk.SKINNY_OPT_FORCE_STAGES, 17), (sk.SKINNY_OPT_WAIT_TIMEOUT_US, -1),
                                     (sk.SKINNY_OPT_LATE_TRIGGER, 2), (sk.SKINNY_OPT_FUSE_NORM, 2), (99, 0)])
def test_option_values_are_checked(opt, bad):
    with pytest.raises(sk.SkinnyError):
        sk.skinny_set_option(opt, bad)


def test_late_trigger_option_round_trip():
    """SKINNY_OPT_LATE_TRIGGER is 0 by default, settable to 0 or 1, and the
    options context restores it; it changes no plan (only when a launch lets
    its dependents start)."""
    assert sk.skinny_get_option(sk.SKINNY_OPT_LATE_TRIGGER) == 0
    p0 = plan(8, 7168, 14336)
    with sk.options(late_trigger=1):
        assert sk.skinny_get_option(sk.SKINNY_OPT_LATE_TRIGGER) == 1
        assert plan(8, 7168, 14336) == p0
    assert sk.skinny_get_option(sk.SKINNY_OPT_LATE_TRIGGER) == 0


def test_every_workload_case_has_a_plan():
    import skinny_inputs as si
    for c in si.iter_all():
        p = plan(c.M, c.N, c.K, ldy=c.ly)
        assert p["smem_bytes"] <= 227 * 1024
        assert p["grid_x"] >= 1 and p["grid_y"] >= 1


def _table_entries():
    path = os.path.join(ROOT, "latency_skinny_bf16_gb300", "csrc", "tuning_table.inc")
    out = []
    with open(path) as f:
        for line in f:
            line = line.split("//", 1)[0].strip()
            if line.startswith("{"):
                vals = [int(v) for v in line.strip("{},").split(",")]
                out.append(vals)
    return out


def test_every_tuned_entry_is_a_supported_plan_and_is_used():
    for K, N, m_lo, m_hi, be, co, s, bn, st, bk, cl in _table_entries():
        assert 1 <= m_lo <= m_hi <= 64
        # a row never spans two kernels: 1..8 / 9..16 / 17..32 / 33..64 tokens
        assert (m_lo <= 8) == (m_hi <= 8) and (m_lo <= 16) == (m_hi <= 16) and (m_lo <= 32) == (m_hi <= 32)
        if m_hi > 16:   # tensor cores only: split-K MMA, the tensor-core dot-product or tcgen05
            assert (co == sk.SKINNY_CONSUMER_MMA and be in (sk.SKINNY_BACKEND_SPLITK, sk.SKINNY_BACKEND_DOTPROD)) \
                or be == sk.SKINNY_BACKEND_TCGEN05
        for M in range(m_lo, m_hi + 1):
            p = plan(M, N, K)
            assert p["tuned"] == 1, (K, N, M)
            assert p["backend"] == be
            if be == sk.SKINNY_BACKEND_SPLITK:
                assert (p["consumer"], p["split_k"]) == (co, s)
                if st:
                    assert p["stages"] == st
                if bk:
                    assert p["stage_k"] == bk
            elif be == sk.SKINNY_BACKEND_TCGEN05:
                assert (p["split_k"], p["consumer"]) == (s, sk.SKINNY_CONSUMER_MMA)
                assert (bn == 0 or p["block_n"] == bn) and (cl == 0 or p["grid_y"] == cl)
                check_tc_geometry(p, M, N, K)
                if st:
                    assert p["stages"] == st
                if bk:
                    assert p["stage_k"] == bk
            elif be == sk.SKINNY_BACKEND_STREAM:
                assert (p["consumer"], p["block_n"], p["grid_y"]) == (sk.SKINNY_CONSUMER_MMA, 16, 1)
                if bk:
                    assert p["stage_k"] == bk
            else:
                assert p["block_n"] == bn and p["consumer"] == (co if co else sk.SKINNY_CONSUMER_FMA)
            assert p["smem_bytes"] <= 227 * 1024


def test_forced_gpu_test_plans_fit_on_gb300():
    """Every forced persistent split-K configuration the GPU tests run plans on a
    152-SM GB300 (so a GPU run never spends its time on a refused plan)."""
    import test_parity_gpu as tp
    for cons in (sk.SKINNY_CONSUMER_FMA, sk.SKINNY_CONSUMER_MMA):
        for split, clusters, stages, stage_k in tp.PERSISTENT_CFGS:
            c = tp.persistent_case(cons, split)
            with sk.options(backend=sk.SKINNY_BACKEND_SPLITK, consumer=cons, split_k=split, clusters=clusters,
                            stages=stages, stage_k=stage_k):
                p = plan(c.M, c.N, c.K, ldy=c.N + 9)
            assert (p["grid_x"], p["grid_y"]) == (split, clusters)


def test_projection_shapes_at_large_m_take_a_fitting_splitk_plan():
    # a one-shot ring that would not fit shared memory is shortened, not dropped
    for (N, K) in ((7168, 14336), (2112, 7168)):
        for M in (5, 8, 16):
            with sk.options(backend=sk.SKINNY_BACKEND_SPLITK):
                p = plan(M, N, K, ldy=N + 64)
            assert p["backend"] == sk.SKINNY_BACKEND_SPLITK and p["smem_bytes"] <= 227 * 1024


@pytest.mark.parametrize("kw,expect", [
    (dict(Y=C16 + 1), sk.SKINNY_ERR_MISALIGNED),      # bf16 Y: 2-byte alignment
    (dict(Y=B16 + 1024), sk.SKINNY_ERR_INVALID_VALUE),  # overlaps W (2-byte elements)
    (dict(M=65), sk.SKINNY_ERR_UNSUPPORTED),
    (dict(ldy=31), sk.SKINNY_ERR_INVALID_VALUE),
    (dict(M=0), sk.SKINNY_OK),
])
def test_bf16_output_argument_errors(kw, expect):
    args = dict(X=A16, ldx=64, W=B16, ldw=64, Y=C16, ldy=32, M=4, N=32, K=64)
    args.update(kw)
    assert sk.skinny_gemm_bf16_bf16out(args["X"], args["ldx"], args["W"], args["ldw"], args["Y"], args["ldy"],
                                       args["M"], args["N"], args["K"], 0) == expect


def test_bf16_output_two_byte_aligned_y_passes_the_checks():
    # C16 + 2 is misaligned for fp32 Y but fine for bf16 Y
    assert call(Y=C16 + 2) == sk.SKINNY_ERR_MISALIGNED
    st = sk.skinny_gemm_bf16_bf16out(A16, 64, B16, 64, C16 + 2, 32, 4, 32, 64, 0)
    assert st in (sk.SKINNY_OK, sk.SKINNY_ERR_NO_DEVICE)


# ---------------------------------------------------------------- 17..64 tokens
MID_M = (17, 24, 32, 33, 40, 48, 63, 64)


def test_mid_m_takes_a_tensor_core_path():
    for M in MID_M:
        for (N, K) in ((256, 7168), (384, 7168), (2112, 7168), (1536, 4096), (7168, 14336)):
            p = plan(M, N, K)
            assert p["consumer"] == sk.SKINNY_CONSUMER_MMA and p["smem_bytes"] <= 227 * 1024, (M, N, K)
            if p["backend"] == sk.SKINNY_BACKEND_SPLITK:
                assert p["block_n"] == 16
                assert p["split_k"] * p["k_chunk"] >= K and p["k_chunk"] % 16 == 0
                if p["split_k"] > 1:
                    # a single partial-sum buffer: no cluster loops over two tiles
                    assert p["grid_y"] == (N + 15) // 16
            elif p["backend"] == sk.SKINNY_BACKEND_TCGEN05:
                check_tc_geometry(p, M, N, K)
            else:
                assert p["backend"] == sk.SKINNY_BACKEND_DOTPROD and p["block_n"] in (16, 32, 64)
                assert 2 * N * K >= 16e6 and p["k_chunk"] % 32 == 0
    # the default rule on untuned shapes: split-K below 16 MB of W, tcgen05 above
    assert plan(40, 320, 7168)["backend"] == sk.SKINNY_BACKEND_SPLITK
    p = plan(40, 8192, 4096)
    assert (p["backend"], p["consumer"]) == (sk.SKINNY_BACKEND_TCGEN05, sk.SKINNY_CONSUMER_MMA)
    # 1024 row groups: one range per CTA slot would give tiles of 32 rows (too
    # few W bytes per MMA); the cost model takes clusters of 2 (152 ranges of
    # 6-7 groups: tiles of up to 56 rows, two CTAs on every SM)
    assert (p["split_k"], p["stage_k"], p["grid_y"], p["block_n"]) == (2, 128, 152, 64)
    check_tc_geometry(p, 40, 8192, 4096)
    # 9..16 tokens on large weights take it too; fewer stay on the earlier backends
    assert plan(12, 8192, 4096)["backend"] == sk.SKINNY_BACKEND_TCGEN05
    assert plan(8, 8192, 3072)["backend"] == sk.SKINNY_BACKEND_DOTPROD
    with sk.options(backend=sk.SKINNY_BACKEND_DOTPROD):
        assert plan(20, 320, 7168)["consumer"] == sk.SKINNY_CONSUMER_MMA


def test_mid_m_unsupported_shapes_are_refused_on_the_host():
    # 7 MB of W: the split-K X slice of 64 tokens does not fit; tcgen05 takes it
    assert plan(64, 256, 14336)["backend"] == sk.SKINNY_BACKEND_TCGEN05
    assert plan(64, 7168, 14336)["backend"] == sk.SKINNY_BACKEND_TCGEN05   # 206 MB of W, tuned
    with sk.options(backend=sk.SKINNY_BACKEND_DOTPROD):
        p = plan(64, 7168, 14336)                  # the tensor-core dot-product stages X in chunks
    assert p["backend"] == sk.SKINNY_BACKEND_DOTPROD and p["k_chunk"] < 14336
    with pytest.raises(sk.SkinnyError) as e:
        with sk.options(backend=sk.SKINNY_BACKEND_DOTPROD):
            plan(20, 256, 7184)                    # K % 32 != 0: no tensor-core dot-product
    assert e.value.status == sk.SKINNY_ERR_UNSUPPORTED
    # K % 16 != 0 with 16-byte aligned rows: only the tcgen05 backend
    assert plan(20, 256, 7160)["backend"] == sk.SKINNY_BACKEND_TCGEN05
    with pytest.raises(sk.SkinnyError) as e:
        with sk.options(backend=sk.SKINNY_BACKEND_SPLITK):
            plan(20, 256, 7160)
    assert e.value.status == sk.SKINNY_ERR_UNSUPPORTED
    for kw in (dict(K=7176, W=B16 + 8), dict(K=7169)):   # W rows / X rows not 16-byte aligned
        K = kw.pop("K")
        with pytest.raises(sk.SkinnyError) as e:
            plan(20, 256, K, **kw)
        assert e.value.status == sk.SKINNY_ERR_UNSUPPORTED
    for opts in (dict(backend=sk.SKINNY_BACKEND_DOTPROD, consumer=sk.SKINNY_CONSUMER_FMA),
                 dict(consumer=sk.SKINNY_CONSUMER_FMA),
                 dict(backend=sk.SKINNY_BACKEND_SPLITK, split_k=8, clusters=4)):
        with sk.options(**opts):
            with pytest.raises(sk.SkinnyError) as e:
                plan(40, 256, 7168)
            assert e.value.status == sk.SKINNY_ERR_UNSUPPORTED
    # small M is unchanged by the mid-M rules
    assert plan(16, 256, 7200)["backend"] == sk.SKINNY_BACKEND_SPLITK


def test_mid_m_forced_split_sizes_plan():
    for M in (17, 32, 64):
        for S in (1, 2, 4, 8):
            with sk.options(backend=sk.SKINNY_BACKEND_SPLITK, consumer=sk.SKINNY_CONSUMER_MMA, split_k=S):
                try:
                    p = plan(M, 256, 4096)
                except sk.SkinnyError as e:
                    # only a slice too long for shared memory may refuse
                    # (32 tokens x 4096 x 2 B = 256 KB at S = 1; 64 tokens x 2048 x 2 B at S = 2)
                    assert e.status == sk.SKINNY_ERR_UNSUPPORTED and (S == 1 or (M > 32 and S == 2))
                    continue
            assert p["split_k"] == S and p["smem_bytes"] <= 227 * 1024


# ---------------------------------------------------------------- K-outer streaming backend
def test_stream_plan_for_large_weights_with_long_k():
    with sk.options(backend=sk.SKINNY_BACKEND_STREAM):
        p = plan(16, 8192, 8192)             # 128 MB of W
    assert (p["backend"], p["consumer"]) == (sk.SKINNY_BACKEND_STREAM, sk.SKINNY_CONSUMER_MMA)
    tiles = 8192 // 16
    assert p["grid_x"] == 152 and p["grid_y"] == 1 and p["split_k"] == 1
    per = -(-tiles // p["grid_x"])
    assert per <= 4 and p["stages"] >= per + 1 and p["smem_bytes"] <= 227 * 1024
    assert p["stage_k"] % 64 == 0 and p["stage_k"] <= 2048 and p["k_chunk"] == 8192
    # K split into equal chunks of at most 2048 elements
    assert -(-8192 // p["stage_k"]) * p["stage_k"] - 8192 < 64


def test_stream_needs_aligned_x_and_w_and_k16():
    for kw in (dict(X=A16 + 2), dict(ldx=8200 + 1), dict(W=B16 + 8)):
        p = plan(16, 8192, 8192, **kw)
        assert p["backend"] != sk.SKINNY_BACKEND_STREAM
    with sk.options(backend=sk.SKINNY_BACKEND_STREAM):
        for kw in (dict(X=A16 + 2), dict(W=B16 + 8)):
            with pytest.raises(sk.SkinnyError) as e:
                plan(8, 8192, 8192, **kw)
            assert e.value.status == sk.SKINNY_ERR_UNSUPPORTED
        with pytest.raises(sk.SkinnyError):
            plan(8, 256, 7176)               # K % 16 != 0
        with pytest.raises(sk.SkinnyError):
            plan(17, 256, 7168)              # M > 16
        with sk.options(consumer=sk.SKINNY_CONSUMER_FMA):
            with pytest.raises(sk.SkinnyError):
                plan(8, 256, 7168)


def test_stream_forced_shapes_plan():
    # small weights, forced: clusters = CTAs, every CTA at most 4 tiles
    with sk.options(backend=sk.SKINNY_BACKEND_STREAM, clusters=5):
        p = plan(3, 16 * 13 + 5, 4096)
        assert p["grid_x"] == 5 and p["stages"] >= 4
    with sk.options(backend=sk.SKINNY_BACKEND_STREAM, clusters=2):
        with pytest.raises(sk.SkinnyError):  # 14 tiles on 2 CTAs: 7 per CTA > 4
            plan(3, 16 * 13 + 5, 4096)
    with sk.options(backend=sk.SKINNY_BACKEND_STREAM, clusters=5, stages=3):
        with pytest.raises(sk.SkinnyError):  # the ring must hold 3 tiles + X + 1
            plan(3, 16 * 13 + 5, 4096)
    with sk.options(backend=sk.SKINNY_BACKEND_STREAM, stage_k=64):
        p = plan(16, 37, 1040)
        assert p["stage_k"] == 64 and p["grid_x"] == 3


# ---------------------------------------------------------------- router epilogue (softmax + top-k)
D16 = 0x7F0030000000


def topk_call(L=C16, ldl=256, M=4, N=256, k=8, renorm=0, Wt=A16, ldw=8, ids=B16, ldid=8):
    return sk.skinny_router_topk(L, ldl, M, N, k, renorm, Wt, ldw, ids, ldid, 0)


@pytest.mark.parametrize("kw,expect", [
    (dict(M=-1), sk.SKINNY_ERR_INVALID_VALUE),
    (dict(N=-1), sk.SKINNY_ERR_INVALID_VALUE),
    (dict(k=-1), sk.SKINNY_ERR_INVALID_VALUE),
    (dict(M=0), sk.SKINNY_OK),
    (dict(k=0), sk.SKINNY_OK),
    (dict(M=0, L=0, Wt=0, ids=0), sk.SKINNY_OK),
    (dict(k=257, ldw=300, ldid=300), sk.SKINNY_ERR_INVALID_VALUE),       # k > N
    (dict(N=8193, ldl=8193), sk.SKINNY_ERR_UNSUPPORTED),
    (dict(k=65, ldw=65, ldid=65), sk.SKINNY_ERR_UNSUPPORTED),
    (dict(M=65536), sk.SKINNY_ERR_UNSUPPORTED),
    (dict(ldl=255), sk.SKINNY_ERR_INVALID_VALUE),
    (dict(ldw=7), sk.SKINNY_ERR_INVALID_VALUE),
    (dict(ldid=7), sk.SKINNY_ERR_INVALID_VALUE),
    (dict(L=0), sk.SKINNY_ERR_INVALID_VALUE),
    (dict(Wt=0), sk.SKINNY_ERR_INVALID_VALUE),
    (dict(ids=0), sk.SKINNY_ERR_INVALID_VALUE),
    (dict(L=C16 + 2), sk.SKINNY_ERR_MISALIGNED),
    (dict(Wt=A16 + 2), sk.SKINNY_ERR_MISALIGNED),
    (dict(ids=B16 + 1), sk.SKINNY_ERR_MISALIGNED),
    (dict(Wt=C16 + 64), sk.SKINNY_ERR_INVALID_VALUE),                     # weights overlap the logits
    (dict(ids=C16 + 4 * 256 * 3), sk.SKINNY_ERR_INVALID_VALUE),           # ids overlap the logits
    (dict(ids=A16 + 16), sk.SKINNY_ERR_INVALID_VALUE),                    # ids overlap the weights
    (dict(), sk.SKINNY_ERR_NO_DEVICE),                                    # valid: needs a GPU
])
def test_router_topk_argument_errors_are_host_side(kw, expect):
    assert topk_call(**kw) == expect


def test_router_fused_checks_both_steps_before_launching():
    def fused(**kw):
        a = dict(X=A16, ldx=7168, W=B16, ldw=7168, L=C16, ldl=256, M=4, N=256, K=7168, k=8, renorm=1,
                 Wt=D16, ldwt=8, ids=D16 + 4096, ldid=8)
        a.update(kw)
        return sk.skinny_router_bf16_topk(a["X"], a["ldx"], a["W"], a["ldw"], a["L"], a["ldl"], a["M"], a["N"],
                                          a["K"], a["k"], a["renorm"], a["Wt"], a["ldwt"], a["ids"], a["ldid"], 0)
    assert fused() == sk.SKINNY_ERR_NO_DEVICE
    assert fused(M=65) == sk.SKINNY_ERR_UNSUPPORTED                   # GEMM: M > 64
    assert fused(ldx=100) == sk.SKINNY_ERR_INVALID_VALUE              # GEMM: ldx < K
    assert fused(k=100) == sk.SKINNY_ERR_UNSUPPORTED                  # epilogue: k > 64
    assert fused(Wt=B16 + 64) == sk.SKINNY_ERR_INVALID_VALUE          # weights overlap W
    assert fused(ids=A16 + 8) == sk.SKINNY_ERR_INVALID_VALUE          # ids overlap X
    assert fused(L=B16 + 1024) == sk.SKINNY_ERR_INVALID_VALUE         # logits overlap W
    assert fused(M=0) == sk.SKINNY_OK


# ---------------------------------------------------------------- fp32 router weights
def f32w_call(X=A16, ldx=64, W=B16, ldw=64, Y=C16, ldy=32, M=4, N=32, K=64):
    return sk.skinny_gemm_bf16_f32w(X, ldx, W, ldw, Y, ldy, M, N, K, 0)


@pytest.mark.parametrize("kw,expect", [
    (dict(M=-1), sk.SKINNY_ERR_INVALID_VALUE),
    (dict(M=17), sk.SKINNY_ERR_UNSUPPORTED),       # dot-product kernel only: M <= 16
    (dict(M=0), sk.SKINNY_OK),
    (dict(ldw=63), sk.SKINNY_ERR_INVALID_VALUE),
    (dict(W=B16 + 2), sk.SKINNY_ERR_MISALIGNED),    # fp32: 4-byte aligned
    (dict(Y=B16 + 4 * 64 * 31), sk.SKINNY_ERR_INVALID_VALUE),   # Y overlaps the fp32 W (4-byte elements)
    (dict(), sk.SKINNY_ERR_NO_DEVICE),
])
def test_f32w_argument_errors_are_host_side(kw, expect):
    assert f32w_call(**kw) == expect


def _p32(W=B16, ldw=None, M=4, N=256, K=7168):
    return sk.skinny_plan_for_f32w(A16, K, W, ldw or K, C16, N, M, N, K, 152)


def test_f32w_plan_follows_alignment():
    """The CUDA-core kernel below 6 tokens, on weights under 4 MB, or where the
    tensor-core kernel cannot read W (rows not 16-byte aligned, K % 32 != 0):
    W loads as wide as the pointer and ldw allow."""
    FMA = sk.SKINNY_CONSUMER_FMA
    assert _p32(M=5)["vec_elems"] == 4 and _p32(M=5)["consumer"] == FMA
    assert _p32(M=16, N=128, K=2880)["consumer"] == FMA      # 1.5 MB of fp32 W
    for kw, vec in ((dict(W=B16 + 8), 2), (dict(W=B16 + 4), 1), (dict(K=7169), 1), (dict(K=7170), 2),
                    (dict(K=7172), 4)):
        p = _p32(M=8, **kw)
        assert (p["vec_elems"], p["consumer"]) == (vec, FMA), (kw, p)
    assert _p32(M=2, N=2048)["block_n"] == 4 and _p32(M=2, N=2048)["grid_x"] == 512
    with sk.options(consumer=FMA):
        assert _p32(M=16, K=14336)["k_chunk"] % 1024 == 0    # X in chunks: 16 x 14336 bf16 > budget
    assert _p32(M=0)["grid_x"] == 0


def test_f32w_tensor_core_plans():
    """From 6 tokens on weights of 4 MB or more, with 16-byte W rows and
    K % 32 == 0 (or forced): 16-row blocks, K over
    a cluster of S CTAs (the largest power of two up to 8 that keeps the grid
    within two CTAs per SM and gives every rank some K), the rank's X slice
    resident, 8 warps up to 8 tokens and 4 above; forced consumer / split /
    block honoured; refused where the kernel cannot run."""
    MMA = sk.SKINNY_CONSUMER_MMA
    for (M, N, K, S, force) in ((6, 256, 7168, 8, 0), (16, 384, 7168, 8, 0), (16, 128, 2880, 8, MMA),
                                (8, 2112, 7168, 2, 0)):
        with sk.options(consumer=force):
            p = _p32(M=M, N=N, K=K)
        blocks = -(-N // 16)
        ks = -(-(-(-K // S)) // 32) * 32
        assert (p["consumer"], p["block_n"], p["split_k"], p["vec_elems"]) == (MMA, 16, S, 4), p
        assert (p["grid_x"], p["grid_y"]) == ((S, blocks) if S > 1 else (blocks, 1))
        assert p["k_chunk"] == ks and (S - 1) * ks < K
        assert blocks * S <= 2 * 152 and p["smem_bytes"] <= 227 * 1024
        assert p["threads"] == (256 if M <= 8 else 128)
    with sk.options(consumer=MMA, split_k=4, block_n=32):
        p = _p32(M=2)
        assert (p["consumer"], p["split_k"], p["block_n"], p["grid_x"], p["grid_y"]) == (MMA, 4, 32, 4, 8)
    with sk.options(consumer=MMA):
        for kw in (dict(W=B16 + 8), dict(K=7170), dict(K=7172), dict(K=16)):
            with pytest.raises(sk.SkinnyError) as e:
                _p32(**kw)
            assert e.value.status == sk.SKINNY_ERR_UNSUPPORTED
        with sk.options(split_k=8):
            with pytest.raises(sk.SkinnyError):
                _p32(K=224)                                   # 8 slices of 32: the last rank gets none


# ---------------------------------------------------------------- RMS norm + q_b GEMM
E16 = 0x7F0040000000


def norm_call(X=A16, ldx=64, G=D16, eps=1e-6, XN=E16, ldxn=64, W=B16, ldw=64, Y=C16, ldy=32, M=4, N=32, K=64):
    return sk.skinny_rmsnorm_gemm_bf16(X, ldx, G, eps, XN, ldxn, W, ldw, Y, ldy, M, N, K, 0)


@pytest.mark.parametrize("kw,expect", [
    (dict(M=-1), sk.SKINNY_ERR_INVALID_VALUE),
    (dict(M=0), sk.SKINNY_OK),
    (dict(M=65), sk.SKINNY_ERR_UNSUPPORTED),
    (dict(eps=-1.0), sk.SKINNY_ERR_INVALID_VALUE),
    (dict(eps=float("inf")), sk.SKINNY_ERR_INVALID_VALUE),
    (dict(eps=float("nan")), sk.SKINNY_ERR_INVALID_VALUE),
    (dict(G=0), sk.SKINNY_ERR_INVALID_VALUE),
    (dict(X=0), sk.SKINNY_ERR_INVALID_VALUE),
    (dict(ldx=63), sk.SKINNY_ERR_INVALID_VALUE),
    (dict(ldxn=63), sk.SKINNY_ERR_INVALID_VALUE),
    (dict(X=A16 + 1), sk.SKINNY_ERR_MISALIGNED),
    (dict(G=D16 + 1), sk.SKINNY_ERR_MISALIGNED),
    (dict(XN=A16 + 64), sk.SKINNY_ERR_INVALID_VALUE),    # XN overlaps X
    (dict(XN=D16 + 2), sk.SKINNY_ERR_INVALID_VALUE),     # XN overlaps gamma
    (dict(XN=B16 + 64), sk.SKINNY_ERR_INVALID_VALUE),    # XN overlaps W
    (dict(Y=A16 + 128), sk.SKINNY_ERR_INVALID_VALUE),    # Y overlaps X
    (dict(), sk.SKINNY_ERR_NO_DEVICE),
])
def test_rmsnorm_gemm_argument_errors_are_host_side(kw, expect):
    assert norm_call(**kw) == expect


def test_tcgen05_tile_heights():
    for bn in (64, 128):
        with sk.options(backend=sk.SKINNY_BACKEND_TCGEN05, block_n=bn):
            for M, N, K in ((1, 24576, 1536), (40, 2112, 7168), (64, 100, 520)):
                p = plan(M, N, K)
                assert (p["backend"], p["block_n"]) == (sk.SKINNY_BACKEND_TCGEN05, bn)
                check_tc_geometry(p, M, N, K)
    with sk.options(backend=sk.SKINNY_BACKEND_TCGEN05, block_n=32):
        with pytest.raises(sk.SkinnyError):
            plan(8, 24576, 1536)


def test_tcgen05_plans_are_consistent():
    """Every tcgen05 plan the host accepts fits what the kernel assumes: a ring
    of whole stages in the shared memory it asks for (>= 30 KB, so at most 7
    CTAs share an SM's tensor memory), K slices of whole stages covering K, a
    ring large enough to receive the cluster's partials, and the grid the
    launcher checks."""
    import random
    rng = random.Random(11)
    ran = 0
    for _ in range(600):
        M = rng.randint(1, 64)
        N = rng.randint(1, 30000)
        K = 8 * rng.randint(1, 2048)
        bn, S = rng.choice([0, 64, 128]), rng.choice([0, 1, 2, 4, 8])
        bk, st = rng.choice([0, 64, 128, 256]), rng.choice([0, 1, 2, 3, 6])
        with sk.options(backend=sk.SKINNY_BACKEND_TCGEN05, block_n=bn, split_k=S, stage_k=bk, stages=st):
            try:
                p = plan(M, N, K, X=0x100000000000, W=0x200000000000, Y=0x300000000000)   # no overlap
            except sk.SkinnyError as e:
                assert e.status == sk.SKINNY_ERR_UNSUPPORTED
                continue
        ran += 1
        tm, s, sk_ = p["block_n"], p["split_k"], p["stage_k"]
        assert tm in (64, 128) and (bn == 0 or tm == bn) and (S == 0 or s == S) and (bk == 0 or sk_ == bk)
        assert (st == 0 or p["stages"] == st) and 1 <= p["stages"] <= 16
        check_tc_geometry(p, M, N, K)
    assert ran > 300


def test_tcgen05_refuses_rows_a_tensor_map_cannot_address():
    """The tensor maps need 16-byte aligned row starts for X and W (base
    pointers and strides): anything else is refused on the host when tcgen05
    is forced, and planned on another backend when it is not."""
    with sk.options(backend=sk.SKINNY_BACKEND_TCGEN05):
        assert plan(16, 4096, 4096)["backend"] == sk.SKINNY_BACKEND_TCGEN05
        for kw in (dict(X=A16 + 2), dict(W=B16 + 8), dict(ldx=4100), dict(ldw=4100)):
            with pytest.raises(sk.SkinnyError) as e:
                plan(16, 4096, 4096, **kw)
            assert e.value.status == sk.SKINNY_ERR_UNSUPPORTED
    for kw in (dict(X=A16 + 2), dict(ldx=4100)):
        assert plan(16, 4096, 4096, **kw)["backend"] != sk.SKINNY_BACKEND_TCGEN05


def test_pdl_follows_how_the_plan_moves_w():
    """PDL mode 1 puts the attribute on every plan that stages W through shared
    memory (split-K, streaming, tcgen05) and on dot-product plans (W loaded
    into registers through L1) under 16 MB of weight; mode 2 on every call; 0
    on none."""
    dot = dict(backend=sk.SKINNY_BACKEND_DOTPROD, consumer=sk.SKINNY_CONSUMER_MMA)
    with sk.options(pdl=1):
        assert plan(4, 256, 7168)["pdl"] == 1                 # the router: 3.7 MB
        with sk.options(**dot):
            assert plan(4, 256, 7168)["pdl"] == 1
            assert plan(4, 24576, 1536)["pdl"] == 0           # 75 MB into registers
        with sk.options(backend=sk.SKINNY_BACKEND_DOTPROD, consumer=sk.SKINNY_CONSUMER_FMA):
            assert plan(1, 24576, 1536)["pdl"] == 0
        for backend in (sk.SKINNY_BACKEND_SPLITK, sk.SKINNY_BACKEND_TCGEN05, sk.SKINNY_BACKEND_STREAM):
            with sk.options(backend=backend):
                p = plan(4, 24576, 1536)
                assert p["backend"] == backend and p["pdl"] == 1, p
        for M in (1, 16):                                     # 206 MB: split-K / tcgen05
            p = plan(M, 7168, 14336)
            assert p["backend"] != sk.SKINNY_BACKEND_DOTPROD and p["pdl"] == 1, p
    with sk.options(pdl=2, **dot):
        assert plan(4, 24576, 1536)["pdl"] == 1
    with sk.options(pdl=0):
        assert plan(4, 256, 7168)["pdl"] == 0
        assert plan(1, 7168, 14336)["pdl"] == 0


def test_dotmma_cluster_split_plans():
    """K over a cluster of S CTAs on the tensor-core dot-product: grid S x blocks, a K chunk no
    longer than a rank's slice, slot bytes in the shared memory; refused past 16 tokens and
    where a rank would get no K."""
    dm = dict(backend=sk.SKINNY_BACKEND_DOTPROD, consumer=sk.SKINNY_CONSUMER_MMA)
    for (M, N, K, S, bn) in ((16, 256, 7168, 8, 16), (12, 384, 7168, 4, 32), (5, 2112, 7168, 2, 64)):
        with sk.options(split_k=S, block_n=bn, **dm):
            p = plan(M, N, K)
        ks = -(-(-(-K // S)) // 32) * 32
        assert (p["backend"], p["consumer"], p["split_k"], p["block_n"]) == (1, 2, S, bn)
        assert (p["grid_x"], p["grid_y"]) == (S, -(-N // bn))
        assert p["k_chunk"] % 32 == 0 and p["k_chunk"] <= ks and (S - 1) * ks < K
        mt = 8 if M <= 8 else 16
        assert p["smem_bytes"] >= S * bn * mt * 4 + mt * p["k_chunk"] * 2
    for (M, N, K, S) in ((17, 256, 7168, 2), (8, 256, 64, 8), (16, 256, 96, 4)):
        with sk.options(split_k=S, **dm):
            with pytest.raises(sk.SkinnyError):
                plan(M, N, K)


def test_tuned_shapes_cover_every_small_m():
    """A shape in the tuning table has a line for every M = 1..16: a partial re-tune that
    dropped lines would send the missing token counts to the untuned default rule."""
    ranges = {}
    for K, N, m_lo, m_hi, *_ in _table_entries():
        ranges.setdefault((K, N), []).append((m_lo, m_hi))
    for shape, rs in ranges.items():
        covered = set()
        for lo, hi in rs:
            covered.update(range(lo, hi + 1))
        assert set(range(1, 17)) <= covered, (shape, sorted(set(range(1, 17)) - covered))
