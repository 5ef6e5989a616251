"""Pins for the CPU oracle: results that do not come from the oracle itself.

Each test checks the oracle against something the pages or the mathematics fix:
hand-worked golden values (``tests/golden/``), exact rational brute force on
tiny inputs, closed forms (one-hot rows, identity weights, K = 1), invariants
(power-of-two scaling, additivity, row independence, zero-padding of K,
strides), special values, and a float64 library matmul.  The last test plants
mistakes in a copy of the oracle's C source and checks that the pins catch
every one of them.
"""
import math
import os
import random
import struct
import subprocess
import tempfile
from fractions import Fraction

import numpy as np
import pytest

import oracle
import skinny_inputs as si

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


# ----------------------------------------------------------------------------- helpers

def exact_bits(value: float) -> int:
    """bf16 bits of a value that bf16 represents exactly (asserts so)."""
    (word,) = struct.unpack("<I", struct.pack("<f", float(value)))
    assert word & 0xFFFF == 0, f"{value!r} is not exactly representable in bf16"
    return word >> 16


def bits_to_fraction(bits: int) -> Fraction:
    """Exact rational value of a finite bf16 pattern, from the format definition."""
    sign = -1 if bits & 0x8000 else 1
    exp = (bits >> 7) & 0xFF
    man = bits & 0x7F
    assert exp != 0xFF
    if exp == 0:
        return sign * Fraction(man, 128) * Fraction(1, 2 ** 126)
    return sign * (1 + Fraction(man, 128)) * (Fraction(2) ** (exp - 127))


def random_grid_bits(rng: random.Random, n: int, emin: int = -4, emax: int = 4) -> np.ndarray:
    """bf16 values s * (1 + j/128) * 2^e with e in [emin, emax] (or zero)."""
    out = np.empty(n, np.uint16)
    for i in range(n):
        if rng.random() < 0.05:
            out[i] = 0
            continue
        s = rng.randrange(2)
        e = rng.randint(emin, emax)
        j = rng.randrange(128)
        out[i] = (s << 15) | ((e + 127) << 7) | j
    return out


def exact_gemm(X, W, M, N, K):
    Xq = [[bits_to_fraction(int(X[m * K + k])) for k in range(K)] for m in range(M)]
    Wq = [[bits_to_fraction(int(W[n * K + k])) for k in range(K)] for n in range(N)]
    Y = [[sum((Xq[m][k] * Wq[n][k] for k in range(K)), Fraction(0)) for n in range(N)]
         for m in range(M)]
    A = [[sum((abs(Xq[m][k] * Wq[n][k]) for k in range(K)), Fraction(0)) for n in range(N)]
         for m in range(M)]
    return Y, A


def parse_worked_examples(path):
    examples = []
    cur = None
    with open(path) as f:
        for raw in f:
            line = raw.split("#", 1)[0].strip()
            if not line:
                continue
            head, *rest = line.split(None, 1)
            if head == "begin":
                cur = {"name": rest[0]}
            elif head == "end":
                examples.append(cur)
                cur = None
            elif head in ("M", "N", "K"):
                cur[head] = int(rest[0])
            else:
                rows = [[float(t) for t in r.split()] for r in rest[0].split(";")]
                cur[head] = rows
    return examples


# ----------------------------------------------------------------------------- golden

def test_bf16_decode_golden():
    n = 0
    with open(os.path.join(GOLDEN, "bf16_decode.txt")) as f:
        for raw in f:
            line = raw.split("#", 1)[0].strip()
            if not line:
                continue
            hx, val = line.split()
            bits = int(hx, 16)
            got = oracle.bf16_to_f64(bits)
            want = float(val)
            if math.isnan(want):
                assert math.isnan(got), hx
            else:
                assert got == want, (hx, got, want)
                assert math.copysign(1.0, got) == math.copysign(1.0, want), hx
            n += 1
    assert n >= 15


@pytest.mark.parametrize("ex", parse_worked_examples(os.path.join(GOLDEN, "worked_examples.txt")),
                         ids=lambda e: e["name"])
def test_worked_examples_golden(ex):
    M, N, K = ex["M"], ex["N"], ex["K"]
    X = np.array([exact_bits(v) for row in ex["X"] for v in row], np.uint16)
    W = np.array([exact_bits(v) for row in ex["W"] for v in row], np.uint16)
    assert X.size == M * K and W.size == N * K
    Y, A = oracle.gemm(X, W, M, N, K)
    assert Y.tolist() == ex["Y"]
    assert A.tolist() == ex["A"]


# ----------------------------------------------------------------------------- brute force

@pytest.mark.parametrize("seed", range(40))
def test_bruteforce_exact_on_tiny_grid_inputs(seed):
    """Tiny shapes, values on a bounded exponent grid: every partial sum is a
    multiple of 2^-22 below 2^16, so fp64 is exact in any order and the oracle
    must equal the rational brute force exactly."""
    rng = random.Random(seed)
    M, N = rng.randint(1, 4), rng.randint(1, 4)
    K = rng.randint(1, 4) if seed < 20 else rng.randint(5, 64)
    X = random_grid_bits(rng, M * K)
    W = random_grid_bits(rng, N * K)
    Y, A = oracle.gemm(X, W, M, N, K)
    Ye, Ae = exact_gemm(X, W, M, N, K)
    for m in range(M):
        for n in range(N):
            assert Fraction(Y[m, n]) == Ye[m][n], (m, n)
            assert Fraction(A[m, n]) == Ae[m][n], (m, n)


@pytest.mark.parametrize("seed", range(10))
def test_bruteforce_within_fp64_bound_on_wide_range(seed):
    """Unrestricted bf16 magnitudes (outlier workload recipe): the oracle is the
    exact sum up to fp64 recursive-summation error, |err| <= K * 2^-53 * A."""
    case = si.Case("bf", M=3, N=3, K=48, seed=1000 + seed, x_dist="normal",
                   w_dist="normal", outliers=True)
    X, W = si.make_inputs(case)
    Y, A = oracle.gemm(X, W, 3, 3, 48)
    Ye, Ae = exact_gemm(X.reshape(-1), W.reshape(-1), 3, 3, 48)
    for m in range(3):
        for n in range(3):
            err = abs(Fraction(Y[m, n]) - Ye[m][n])
            assert err <= Fraction(48) * Fraction(1, 2 ** 53) * Ae[m][n]
            assert abs(Fraction(A[m, n]) - Ae[m][n]) <= Fraction(48) * Fraction(1, 2 ** 53) * Ae[m][n]


# ----------------------------------------------------------------------------- closed forms

def test_one_hot_rows_reproduce_weight_columns():
    case = si.Case("oh", M=1, N=37, K=29, seed=7)
    _, W = si.make_inputs(case)
    K, N = 29, 37
    for k in (0, 1, 13, 28):
        X = np.zeros(K, np.uint16)
        X[k] = exact_bits(1.0)
        Y, _ = oracle.gemm(X, W, 1, N, K)
        for n in range(N):
            assert Y[0, n] == oracle.bf16_to_f64(int(W[n, k]))


def test_identity_weight_reproduces_x():
    K = 23
    case = si.Case("id", M=5, N=K, K=K, seed=8)
    X, _ = si.make_inputs(case)
    W = np.zeros((K, K), np.uint16)
    for i in range(K):
        W[i, i] = exact_bits(1.0)
    Y, _ = oracle.gemm(X, W, 5, K, K)
    for m in range(5):
        for k in range(K):
            assert Y[m, k] == oracle.bf16_to_f64(int(X[m, k]))


def test_k_equals_one_is_a_single_product():
    case = si.Case("k1", M=4, N=9, K=1, seed=9)
    X, W = si.make_inputs(case)
    Y, A = oracle.gemm(X, W, 4, 9, 1)
    for m in range(4):
        for n in range(9):
            p = Fraction(oracle.bf16_to_f64(int(X[m, 0]))) * Fraction(oracle.bf16_to_f64(int(W[n, 0])))
            assert Fraction(Y[m, n]) == p
            assert Fraction(A[m, n]) == abs(p)


# ----------------------------------------------------------------------------- invariants

def _scale_bits_pow2(bits: np.ndarray, j: int) -> np.ndarray:
    """Multiply normal bf16 values by 2^j by moving the exponent field."""
    b = bits.astype(np.int32)
    exp = (b >> 7) & 0xFF
    nz = exp != 0
    assert np.all((exp[nz] + j > 0) & (exp[nz] + j < 255))
    out = np.where(nz, b + (j << 7), b)
    return out.astype(np.uint16)


def test_power_of_two_scaling_is_exact():
    case = si.Case("sc", M=3, N=11, K=300, seed=10)
    X, W = si.make_inputs(case)
    X = np.where(((X >> 7) & 0xFF) == 0, np.uint16(0), X).astype(np.uint16)
    Y, _ = oracle.gemm(X, W, 3, 11, 300)
    for j in (-5, 3, 17):
        Ys, _ = oracle.gemm(_scale_bits_pow2(X, j), W, 3, 11, 300)
        assert np.array_equal(Ys, Y * (2.0 ** j))


def test_additivity():
    """X1 + X2 representable (small integers): Y(X1+X2) = Y(X1) + Y(X2) up to fp64 rounding."""
    rng = np.random.default_rng(11)
    M, N, K = 3, 17, 200
    x1 = rng.integers(-64, 65, size=(M, K))
    x2 = rng.integers(-64, 65, size=(M, K))
    X1 = np.array([exact_bits(v) for v in x1.reshape(-1)], np.uint16)
    X2 = np.array([exact_bits(v) for v in x2.reshape(-1)], np.uint16)
    X12 = np.array([exact_bits(v) for v in (x1 + x2).reshape(-1)], np.uint16)
    _, W = si.make_inputs(si.Case("ad", M=1, N=N, K=K, seed=12))
    Y1, A1 = oracle.gemm(X1, W, M, N, K)
    Y2, A2 = oracle.gemm(X2, W, M, N, K)
    Y12, _ = oracle.gemm(X12, W, M, N, K)
    bound = 3 * K * 2.0 ** -53 * (A1 + A2)
    assert np.all(np.abs(Y12 - (Y1 + Y2)) <= bound)


def test_row_independence_bit_exact():
    case = si.Case("ri", M=6, N=40, K=513, seed=13)
    X, W = si.make_inputs(case)
    Y, _ = oracle.gemm(X, W, 6, 40, 513)
    for m in range(6):
        Ym, _ = oracle.gemm(X[m:m + 1], W, 1, 40, 513)
        assert np.array_equal(Ym[0], Y[m])


def test_zero_padding_of_k_is_bit_exact():
    case = si.Case("zp", M=4, N=21, K=333, seed=14)
    X, W = si.make_inputs(case)
    Y, A = oracle.gemm(X, W, 4, 21, 333)
    for p in (1, 7, 64):
        Xp = np.concatenate([X, np.zeros((4, p), np.uint16)], axis=1)
        Wp = np.concatenate([W, np.zeros((21, p), np.uint16)], axis=1)
        Yp, Ap = oracle.gemm(Xp, Wp, 4, 21, 333 + p)
        assert np.array_equal(Yp, Y) and np.array_equal(Ap, A)


def test_strides_match_compact_and_leave_gaps():
    case = si.Case("st", M=5, N=13, K=77, seed=15)
    X, W = si.make_inputs(case)
    Y, A = oracle.gemm(X, W, 5, 13, 77)
    ldx, ldw, ldy = 77 + 5, 77 + 3, 13 + 9
    Xs = si.embed_rows(X, ldx, fill=0x7FC0)   # NaN in the gaps: must never be read
    Ws = si.embed_rows(W, ldw, fill=0x7FC0)
    sentinel = np.full((5, ldy), -12345.0)
    Ys, As = oracle.gemm(Xs, Ws, 5, 13, 77, ldx=ldx, ldw=ldw, ldy=ldy, Y_init=sentinel)
    assert np.array_equal(Ys[:, :13], Y)
    assert np.array_equal(As[:, :13], A)
    assert np.all(Ys[:, 13:] == -12345.0)


def test_abs_companion_is_abs_gemm():
    case = si.Case("ab", M=3, N=19, K=250, seed=16)
    X, W = si.make_inputs(case)
    Y, A = oracle.gemm(X, W, 3, 19, 250)
    Yabs, _ = oracle.gemm(X & np.uint16(0x7FFF), W & np.uint16(0x7FFF), 3, 19, 250)
    assert np.array_equal(A, Yabs)
    assert np.all(np.abs(Y) <= A)


def test_matches_float64_library_matmul():
    case = si.Case("mm", M=16, N=64, K=1000, seed=17)
    X, W = si.make_inputs(case)
    Xd = (X.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    Wd = (W.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    ref = Xd @ Wd.T
    Y, A = oracle.gemm(X, W, 16, 64, 1000)
    assert np.all(np.abs(Y - ref) <= 2 * 1000 * 2.0 ** -53 * A)


def test_special_values_propagate():
    inf, nan = exact_bits(float("inf")), 0x7FC0
    one, zero, two = exact_bits(1.0), exact_bits(0.0), exact_bits(2.0)
    X = np.array([inf, one, nan, two], np.uint16)          # M=2, K=2
    W = np.array([one, one, zero, one, one, zero], np.uint16)  # N=3, K=2
    Y, _ = oracle.gemm(X, W, 2, 3, 2)
    assert Y[0, 0] == float("inf")        # inf*1 + 1*1
    assert math.isnan(Y[0, 1])            # inf*0 -> NaN
    assert Y[0, 2] == float("inf")        # inf*1 + 1*0
    assert all(math.isnan(v) for v in Y[1])  # NaN row


def test_degenerate_sizes():
    X = np.zeros(4, np.uint16)
    W = np.zeros(4, np.uint16)
    Y, _ = oracle.gemm(X, W, 0, 4, 1)
    assert Y.shape == (0, 4)
    Y, _ = oracle.gemm(X, W, 2, 0, 2, ldy=3, Y_init=np.full((2, 3), 5.0))
    assert np.all(Y == 5.0)
    Y, A = oracle.gemm(X, W, 2, 2, 0)
    assert np.all(Y == 0.0) and np.all(A == 0.0)


def test_points_match_full():
    case = si.Case("pt", M=7, N=50, K=900, seed=18)
    X, W = si.make_inputs(case)
    Y, A = oracle.gemm(X, W, 7, 50, 900)
    rng = np.random.default_rng(0)
    rows = rng.integers(0, 7, 40)
    cols = rng.integers(0, 50, 40)
    y, a = oracle.gemm_points(X, W, 900, rows, cols)
    assert np.array_equal(y, Y[rows, cols]) and np.array_equal(a, A[rows, cols])


# ----------------------------------------------------------------------------- planted mistakes

def _pins_pass(lib) -> bool:
    """A compact subset of the pins above, run against a given oracle build."""
    try:
        for ex in parse_worked_examples(os.path.join(GOLDEN, "worked_examples.txt")):
            M, N, K = ex["M"], ex["N"], ex["K"]
            X = np.array([exact_bits(v) for row in ex["X"] for v in row], np.uint16)
            W = np.array([exact_bits(v) for row in ex["W"] for v in row], np.uint16)
            Y, A = oracle.gemm(X, W, M, N, K, lib=lib)
            if Y.tolist() != ex["Y"] or A.tolist() != ex["A"]:
                return False
        with open(os.path.join(GOLDEN, "bf16_decode.txt")) as f:
            for raw in f:
                line = raw.split("#", 1)[0].strip()
                if not line:
                    continue
                hx, val = line.split()
                got, want = oracle.bf16_to_f64(int(hx, 16), lib=lib), float(val)
                if not (math.isnan(got) and math.isnan(want)) and got != want:
                    return False
        rng = random.Random(5)
        for _ in range(5):
            M, N, K = rng.randint(1, 4), rng.randint(1, 4), rng.randint(1, 40)
            X, W = random_grid_bits(rng, M * K), random_grid_bits(rng, N * K)
            Y, _ = oracle.gemm(X, W, M, N, K, lib=lib)
            Ye, _ = exact_gemm(X, W, M, N, K)
            if any(Fraction(Y[m, n]) != Ye[m][n] for m in range(M) for n in range(N)):
                return False
        case = si.Case("pm", M=3, N=7, K=30, seed=3)
        X, W = si.make_inputs(case)
        ldx, ldw, ldy = 33, 31, 9
        Ys, _ = oracle.gemm(si.embed_rows(X, ldx), si.embed_rows(W, ldw), 3, 7, 30,
                            ldx=ldx, ldw=ldw, ldy=ldy, Y_init=np.zeros((3, ldy)), lib=lib)
        Yc, _ = oracle.gemm(X, W, 3, 7, 30, lib=lib)
        if not np.array_equal(Ys[:, :7], Yc) or np.any(Ys[:, 7:] != 0):
            return False
        return True
    except Exception:
        return False


MUTATIONS = [
    ("drop last k", "for (int k = 0; k < K; ++k) {\n                double prod = skinny_oracle_bf16_to_f64(xrow[k])",
     "for (int k = 0; k < K - 1; ++k) {\n                double prod = skinny_oracle_bf16_to_f64(xrow[k])"),
    ("transposed W index", "const uint16_t *wrow = W + (int64_t)n * ldw;\n            double sum",
     "const uint16_t *wrow = W + (int64_t)n;\n            double sum"),
    ("sign flip", "sum += prod;\n                abs_sum", "sum -= prod;\n                abs_sum"),
    ("fp32 accumulator", "double sum = 0.0;\n            double abs_sum = 0.0;\n            for (int k = 0; k < K; ++k) {\n                double prod",
     "float sum = 0.0f;\n            double abs_sum = 0.0;\n            for (int k = 0; k < K; ++k) {\n                double prod"),
    ("wrong decode shift", "((uint32_t)bits) << 16", "((uint32_t)bits) << 15"),
    ("x stride ignored", "const uint16_t *xrow = X + (int64_t)m * ldx;\n        for (int n",
     "const uint16_t *xrow = X + (int64_t)m * K;\n        for (int n"),
    ("y stride ignored", "Y[(int64_t)m * ldy + n] = sum;", "Y[(int64_t)m * N + n] = sum;"),
]


def test_planted_mistakes_are_caught():
    """Every planted mistake in a copy of the oracle source fails the pins, and
    the unmodified source passes them."""
    with open(oracle.SOURCE_PATH) as f:
        src = f.read()
    with tempfile.TemporaryDirectory() as td:
        clean_so = os.path.join(td, "clean.so")
        oracle.build(src=oracle.SOURCE_PATH, out=clean_so)
        assert _pins_pass(oracle.load(clean_so))
        for name, old, new in MUTATIONS:
            assert src.count(old) == 1, f"mutation anchor not unique: {name}"
            path = os.path.join(td, "mut.c")
            with open(path, "w") as f:
                f.write(src.replace(old, new))
            so = os.path.join(td, f"mut_{abs(hash(name))}.so")
            oracle.build(src=path, out=so)
            assert not _pins_pass(oracle.load(so)), f"planted mistake not caught: {name}"


# ---------------------------------------------------------------- router epilogue (softmax + top-k)

def test_topk_uniform_logits_closed_form():
    """N equal logits: every probability is 1/N, ties go to the lower index."""
    for N, k in ((8, 3), (256, 8), (5, 5)):
        w, ids = oracle.router_topk(np.full((2, N), 0.75, np.float32), k)
        assert ids.tolist() == [list(range(k))] * 2
        assert np.allclose(w, 1.0 / N, rtol=1e-15, atol=0)
        wr, _ = oracle.router_topk(np.full((1, N), -3.0, np.float32), k, renormalize=True)
        assert np.allclose(wr, 1.0 / k, rtol=1e-15, atol=0)


def test_topk_two_level_logits_closed_form():
    """s logits at c and N - s at c - ln(t): the high ones each carry 1 / (s + (N - s) / t)."""
    N, s, t = 64, 5, 4.0
    L = np.zeros((1, N), np.float32)
    hi = [3, 17, 18, 40, 63]
    L[0, :] = np.float32(2.0 - math.log(t))
    L[0, hi] = 2.0
    w, ids = oracle.router_topk(L, s)
    assert ids[0].tolist() == hi
    lo = float(np.float32(2.0 - math.log(t)))
    expected = 1.0 / (s + (N - s) * math.exp(lo - 2.0))
    assert np.allclose(w, expected, rtol=1e-14, atol=0)


def test_topk_matches_stable_argsort_and_library_softmax():
    """Selection equals numpy's stable sort of the negated logits (ties by
    index); probabilities equal scipy's softmax."""
    special = pytest.importorskip("scipy.special")
    rng = np.random.default_rng(31)
    for N, k in ((256, 8), (384, 8), (37, 37), (1000, 1), (16, 4)):
        L = rng.standard_normal((6, N)).astype(np.float32)
        L[0, 5] = L[0, 7] = L[0, 9] = L[0].max() + 1     # a three-way tie at the top
        L[1, ::3] = np.float32(0.25)                       # many ties in the middle
        for renorm in (False, True):
            w, ids = oracle.router_topk(L, k, renormalize=renorm)
            ref_ids = np.argsort(-L, axis=1, kind="stable")[:, :k]
            assert np.array_equal(ids, ref_ids)
            p = special.softmax(L.astype(np.float64), axis=1)
            ref_w = np.take_along_axis(p, ref_ids, axis=1)
            if renorm:
                ref_w = ref_w / ref_w.sum(axis=1, keepdims=True)
            assert np.allclose(w, ref_w, rtol=1e-13, atol=1e-300)


def test_topk_invariants():
    rng = np.random.default_rng(32)
    # multiples of 2^-10 below 16 in magnitude: adding 64 below keeps every logit exact
    L = (np.round(np.clip(rng.standard_normal((4, 200)) * 3, -15, 15) * 1024) / 1024).astype(np.float32)
    w_all, ids_all = oracle.router_topk(L, 200)
    assert np.allclose(w_all.sum(axis=1), 1.0, rtol=1e-13)               # the full softmax sums to 1
    assert (np.diff(w_all, axis=1) <= 0).all()                            # descending
    assert sorted(ids_all[0].tolist()) == list(range(200))                # a permutation
    w8, ids8 = oracle.router_topk(L, 8)
    assert np.array_equal(ids8, ids_all[:, :8]) and np.array_equal(w8, w_all[:, :8])   # prefix of the full order
    wr, _ = oracle.router_topk(L, 8, renormalize=True)
    assert np.allclose(wr.sum(axis=1), 1.0, rtol=1e-13)
    # shifting every logit by the same exactly representable amount changes nothing
    w_s, ids_s = oracle.router_topk(L + np.float32(64.0), 8)
    assert np.array_equal(ids_s, ids8)
    assert np.allclose(w_s, w8, rtol=1e-12)
    # a row with -inf entries: they get probability 0 and come last
    Li = L[:1].copy()
    Li[0, :100] = -np.inf
    wi, idsi = oracle.router_topk(Li, 120)
    assert (idsi[0, :100] >= 100).all() and (wi[0, 100:] == 0).all()


def test_topk_nan_logits_rank_last_and_make_the_weights_nan():
    """Hand-worked rows.  A NaN logit ranks below every value (-inf included)
    and NaNs among themselves by index; the softmax is IEEE arithmetic, so a
    NaN (or +inf) logit makes every weight of its row NaN; a row without them
    keeps its closed-form softmax."""
    nan, inf = np.nan, np.inf
    L = np.array([[nan, 1.0, -inf, 2.0, nan, 0.5],    # NaN first and mid-row
                  [0.0, 3.0, -1.0, -inf, 2.0, 1.0],   # plain row
                  [1.0, inf, 0.0, -1.0, 2.0, 0.0],    # +inf
                  [nan, nan, nan, nan, nan, nan]], np.float32)
    w, ids = oracle.router_topk(L, 6)
    assert ids.tolist() == [[3, 1, 5, 2, 0, 4], [1, 4, 5, 0, 2, 3], [1, 4, 0, 2, 5, 3], [0, 1, 2, 3, 4, 5]]
    assert np.isnan(w[0]).all() and np.isnan(w[2]).all() and np.isnan(w[3]).all()
    denom = math.exp(-3) + 1 + math.exp(-4) + math.exp(-1) + math.exp(-2)
    expect = [1 / denom, math.exp(-1) / denom, math.exp(-2) / denom, math.exp(-3) / denom,
              math.exp(-4) / denom, 0.0]
    assert np.allclose(w[1], expect, rtol=1e-14, atol=0)
    w2, ids2 = oracle.router_topk(L[:1], 2, renormalize=True)
    assert ids2.tolist() == [[3, 1]] and np.isnan(w2).all()


def _topk_pins_pass(lib) -> bool:
    """A compact subset of the top-k pins, run against a given oracle build."""
    try:
        w, ids = oracle.router_topk(np.full((1, 8), 0.5, np.float32), 3, lib=lib)
        if ids.tolist() != [[0, 1, 2]] or not np.allclose(w, 1 / 8, rtol=1e-15, atol=0):
            return False
        rng = np.random.default_rng(33)
        L = rng.standard_normal((3, 50)).astype(np.float32)
        L[0, 10] = L[0, 20] = L[0].max() + 1
        for renorm in (False, True):
            w, ids = oracle.router_topk(L, 6, renormalize=renorm, lib=lib)
            ref_ids = np.argsort(-L, axis=1, kind="stable")[:, :6]
            e = np.exp(L.astype(np.float64) - L.max(axis=1, keepdims=True).astype(np.float64))
            p = e / e.sum(axis=1, keepdims=True)
            ref_w = np.take_along_axis(p, ref_ids, axis=1)
            if renorm:
                ref_w = ref_w / ref_w.sum(axis=1, keepdims=True)
            if not np.array_equal(ids, ref_ids) or not np.allclose(w, ref_w, rtol=1e-13, atol=0):
                return False
        nan = np.nan
        w, ids = oracle.router_topk(np.array([[nan, 1.0, -np.inf, 2.0, nan]], np.float32), 5, lib=lib)
        if ids.tolist() != [[3, 1, 2, 0, 4]] or not np.isnan(w).all():
            return False
        return True
    except Exception:
        return False


TOPK_MUTATIONS = [
    ("ties to the higher index", "    return n < nb;", "    return n > nb;"),
    ("smallest first", "if (!vnan && v != b) return v > b;", "if (!vnan && v != b) return v < b;"),
    ("NaN ranked first", "if (vnan != bnan) return bnan;", "if (vnan != bnan) return vnan;"),
    ("NaN left to the comparison", "if (vnan != bnan) return bnan;", "if (0) return bnan;"),
    ("no renormalisation", "weights[(int64_t)m * ldwt + i] /= chosen;", "weights[(int64_t)m * ldwt + i] *= 1.0;"),
    ("id off by one", "ids[(int64_t)m * ldid + i] = best;", "ids[(int64_t)m * ldid + i] = best + 1;"),
    ("denominator misses the last logit", "for (int n = 0; n < N; ++n) denom += exp",
     "for (int n = 0; n < N - 1; ++n) denom += exp"),
]


def test_topk_planted_mistakes_are_caught():
    with open(oracle.SOURCE_PATH) as f:
        src = f.read()
    with tempfile.TemporaryDirectory() as td:
        clean_so = os.path.join(td, "clean.so")
        oracle.build(src=oracle.SOURCE_PATH, out=clean_so)
        assert _topk_pins_pass(oracle.load(clean_so))
        for name, old, new in TOPK_MUTATIONS:
            assert src.count(old) == 1, f"mutation anchor not unique: {name}"
            path = os.path.join(td, "mut.c")
            with open(path, "w") as f:
                f.write(src.replace(old, new))
            so = os.path.join(td, f"mut_topk_{abs(hash(name))}.so")
            oracle.build(src=path, out=so)
            assert not _topk_pins_pass(oracle.load(so)), f"planted mistake not caught: {name}"


# ---------------------------------------------------------------- fp32 router weights

def _f32_bits_to_float(bits):
    return np.asarray(bits, np.uint32).view(np.float32)


def test_f32w_equals_bf16_oracle_on_bf16_exact_weights():
    """fp32 weights that are exactly bf16 values give the bf16 oracle's result, bit for bit."""
    for seed, (M, N, K) in enumerate([(1, 7, 33), (4, 16, 257), (16, 3, 1000)]):
        X, W = si.make_inputs(si.Case("fw", M=M, N=N, K=K, seed=2000 + seed, outliers=True))
        Wf = _f32_bits_to_float(W.astype(np.uint32) << 16).reshape(N, K)
        Y32, A32 = oracle.gemm_f32w(X, Wf, M, N, K)
        Y16, A16 = oracle.gemm(X, W, M, N, K)
        assert np.array_equal(Y32, Y16) and np.array_equal(A32, A16)


def _exact_f32w(X, Wf, M, N, K):
    xs = [Fraction(oracle.bf16_to_f64(int(b))) for b in X.reshape(-1)]
    ws = [Fraction(float(v)) for v in Wf.reshape(-1)]
    return [[sum(xs[m * K + k] * ws[n * K + k] for k in range(K)) for n in range(N)] for m in range(M)]


@pytest.mark.parametrize("seed", range(4))
def test_f32w_bruteforce_within_fp64_bound(seed):
    """Full-precision fp32 weights (24-bit significands): the fp64 sum is within
    K * 2^-53 * sum|x w| of the exact rational sum."""
    rng = np.random.default_rng(2100 + seed)
    M, N, K = 2, 3, 29
    X = si._to_bf16_bits(__import__("torch").from_numpy(rng.standard_normal((M, K)).astype(np.float32)))
    Wf = (rng.standard_normal((N, K)) * np.exp(rng.uniform(-8, 8, (N, K)))).astype(np.float32)
    Y, A = oracle.gemm_f32w(X, Wf, M, N, K)
    exact = _exact_f32w(X, Wf, M, N, K)
    for m in range(M):
        for n in range(N):
            assert abs(Fraction(Y[m, n]) - exact[m][n]) <= Fraction(K) * Fraction(2) ** -53 * Fraction(A[m, n])
    # and the weights really carry more than bf16 precision
    assert np.any(Wf.view(np.uint32) & 0xFFFF)


def test_f32w_strides_and_gaps():
    X, W = si.make_inputs(si.Case("fws", M=3, N=5, K=40, seed=2200))
    Wf = np.random.default_rng(1).standard_normal((5, 40)).astype(np.float32)
    ldx, ldw = 43, 41
    Xs = si.embed_rows(X, ldx)
    Ws = np.zeros(5 * ldw, np.float32)
    Ws.reshape(5, ldw)[:, :40] = Wf
    Ys, _ = oracle.gemm_f32w(Xs, Ws, 3, 5, 40, ldx=ldx, ldw=ldw)
    Yc, _ = oracle.gemm_f32w(X, Wf, 3, 5, 40)
    assert np.array_equal(Ys, Yc)


def _f32w_pins_pass(lib) -> bool:
    try:
        rng = np.random.default_rng(2300)
        M, N, K = 2, 3, 17
        X = si._to_bf16_bits(__import__("torch").from_numpy(rng.standard_normal((M, K)).astype(np.float32)))
        Wf = rng.standard_normal((N, K)).astype(np.float32)
        Y, A = oracle.gemm_f32w(X, Wf, M, N, K, lib=lib)
        exact = _exact_f32w(X, Wf, M, N, K)
        for m in range(M):
            for n in range(N):
                if abs(Fraction(Y[m, n]) - exact[m][n]) > Fraction(K) * Fraction(2) ** -53 * Fraction(A[m, n]):
                    return False
        return True
    except Exception:
        return False


def test_f32w_planted_mistakes_are_caught():
    muts = [
        ("weights truncated to bf16", "const double t = skinny_oracle_bf16_to_f64(xr[kk]) * (double)wr[kk];",
         "float wt = wr[kk]; uint32_t wb; memcpy(&wb, &wt, 4); wb &= 0xFFFF0000u; memcpy(&wt, &wb, 4);\n"
         "                const double t = skinny_oracle_bf16_to_f64(xr[kk]) * (double)wt;"),
        ("transposed W index", "const float *wr = W + (int64_t)j * ldw;", "const float *wr = W + (int64_t)j;"),
        ("fp32 product", "const double t = skinny_oracle_bf16_to_f64(xr[kk]) * (double)wr[kk];",
         "const double t = (double)((float)skinny_oracle_bf16_to_f64(xr[kk]) * wr[kk]);"),
        ("drop last k", "for (int kk = 0; kk < K; ++kk) {", "for (int kk = 0; kk < K - 1; ++kk) {"),
    ]
    with open(oracle.SOURCE_PATH) as f:
        src = f.read()
    with tempfile.TemporaryDirectory() as td:
        clean_so = os.path.join(td, "clean.so")
        oracle.build(src=oracle.SOURCE_PATH, out=clean_so)
        assert _f32w_pins_pass(oracle.load(clean_so))
        for name, old, new in muts:
            assert src.count(old) == 1, f"mutation anchor not unique: {name}"
            path = os.path.join(td, "mut.c")
            with open(path, "w") as f:
                f.write(src.replace(old, new))
            so = os.path.join(td, f"mut_f32w_{abs(hash(name))}.so")
            oracle.build(src=path, out=so)
            assert not _f32w_pins_pass(oracle.load(so)), f"planted mistake not caught: {name}"


# ---------------------------------------------------------------- RMS norm prologue of the q_b projection

def _bf16(vals):
    return si._to_bf16_bits(__import__("torch").tensor(np.asarray(vals, np.float32)))


def test_rmsnorm_closed_forms():
    K = 16
    ones = _bf16(np.ones(K))
    # a row of +-2^e, unit gain, eps = 0: r = 2^-e and every output is exactly +-1
    row = np.array([4.0, -4.0] * (K // 2), np.float32)
    xn = oracle.rmsnorm(_bf16(row).reshape(1, K), ones, 0.0, 1, K)
    assert xn.tolist() == [[1.0, -1.0] * (K // 2)]
    # the gain multiplies element by element
    g = _bf16(np.arange(1, K + 1) * 0.5)
    xn = oracle.rmsnorm(_bf16(row).reshape(1, K), g, 0.0, 1, K)
    assert xn.tolist() == [[(0.5 * (k + 1)) * (1 if k % 2 == 0 else -1) for k in range(K)]]
    # a zero row stays zero for any eps > 0
    assert not oracle.rmsnorm(_bf16(np.zeros(K)).reshape(1, K), ones, 1e-6, 1, K).any()
    # eps: a row of ones with eps = 3 gives 1 / sqrt(1 + 3) = 1/2 everywhere
    assert (oracle.rmsnorm(ones.reshape(1, K), ones, 3.0, 1, K) == 0.5).all()


def test_rmsnorm_invariants():
    rng = np.random.default_rng(41)
    M, K = 4, 1536
    X = _bf16(rng.standard_normal((M, K))).reshape(M, K)
    ones = _bf16(np.ones(K))
    xn = oracle.rmsnorm(X, ones, 0.0, M, K)
    assert np.allclose((xn ** 2).mean(axis=1), 1.0, rtol=1e-14)         # unit RMS per row
    # scaling a row by a power of two changes nothing (eps = 0, exact)
    X4 = _bf16(np.asarray(X.view(np.uint16).astype(np.uint32) << 16, np.uint32).view(np.float32) * 4.0).reshape(M, K)
    assert np.array_equal(oracle.rmsnorm(X4, ones, 0.0, M, K), xn)
    # rows are independent, and strides are honoured
    xs = si.embed_rows(X, K + 5)
    assert np.array_equal(oracle.rmsnorm(xs, ones, 1e-6, M, K, ldx=K + 5), oracle.rmsnorm(X, ones, 1e-6, M, K))
    assert np.array_equal(oracle.rmsnorm(X[2:3].copy(), ones, 1e-6, 1, K)[0], oracle.rmsnorm(X, ones, 1e-6, M, K)[2])


def _rms_pins_pass(lib) -> bool:
    try:
        K = 16
        ones = _bf16(np.ones(K))
        row = np.array([4.0, -4.0] * (K // 2), np.float32)
        g = _bf16(np.arange(1, K + 1) * 0.5)
        if oracle.rmsnorm(_bf16(row).reshape(1, K), g, 0.0, 1, K, lib=lib).tolist() != \
                [[(0.5 * (k + 1)) * (1 if k % 2 == 0 else -1) for k in range(K)]]:
            return False
        if not (oracle.rmsnorm(ones.reshape(1, K), ones, 3.0, 1, K, lib=lib) == 0.5).all():
            return False
        return True
    except Exception:
        return False


def test_rmsnorm_planted_mistakes_are_caught():
    muts = [
        ("mean over K - 1", "sqrt(ss / (double)K + eps)", "sqrt(ss / (double)(K - 1) + eps)"),
        ("eps dropped", "sqrt(ss / (double)K + eps)", "sqrt(ss / (double)K)"),
        ("gain of the first element", "skinny_oracle_bf16_to_f64(G[k])", "skinny_oracle_bf16_to_f64(G[0])"),
        ("no gain", "* r * skinny_oracle_bf16_to_f64(G[k])", "* r"),
    ]
    with open(oracle.SOURCE_PATH) as f:
        src = f.read()
    with tempfile.TemporaryDirectory() as td:
        clean_so = os.path.join(td, "clean.so")
        oracle.build(src=oracle.SOURCE_PATH, out=clean_so)
        assert _rms_pins_pass(oracle.load(clean_so))
        for name, old, new in muts:
            assert src.count(old) == 1, f"mutation anchor not unique: {name}"
            path = os.path.join(td, "mut.c")
            with open(path, "w") as f:
                f.write(src.replace(old, new))
            so = os.path.join(td, f"mut_rms_{abs(hash(name))}.so")
            oracle.build(src=path, out=so)
            assert not _rms_pins_pass(oracle.load(so)), f"planted mistake not caught: {name}"
