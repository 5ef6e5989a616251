"""The seeded input generators: deterministic, the documented distributions."""
import numpy as np

import skinny_inputs as si


def _vals(bits):
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def test_same_seed_same_bits():
    c = si.Case("d", M=3, N=100, K=257, seed=42)
    X1, W1 = si.make_inputs(c)
    X2, W2 = si.make_inputs(c)
    assert np.array_equal(X1, X2) and np.array_equal(W1, W2)
    X3, _ = si.make_inputs(si.Case("d", M=3, N=100, K=257, seed=43))
    assert not np.array_equal(X1, X3)


def test_distributions():
    X, W = si.make_inputs(si.Case("n", M=16, N=512, K=1024, seed=1))
    x, w = _vals(X), _vals(W)
    assert abs(x.mean()) < 0.02 and abs(x.std() - 1.0) < 0.02
    assert abs(w.mean()) < 0.001 and abs(w.std() - 0.02) < 0.0005
    _, W = si.make_inputs(si.Case("u", M=1, N=256, K=1536, seed=2, w_dist="uniform_isqrtk"))
    w = _vals(W)
    b = 1 / np.sqrt(1536)
    assert w.max() <= b * (1 + 2 ** -8) and w.min() >= -b * (1 + 2 ** -8)
    assert abs(w.std() - b / np.sqrt(3)) < 0.01 * b


def test_outlier_fraction():
    X, W = si.make_inputs(si.Case("o", M=16, N=1000, K=1000, seed=3, x_dist="normal",
                                  w_dist="normal", outliers=True))
    w = np.abs(_vals(W))
    frac = np.mean(w > 20.0)   # a N(0,1) draw exceeds 20 with negligible probability
    assert 0.007 < frac < 0.011


def test_rounding_is_nearest_even():
    import torch
    v = torch.tensor([1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -(1.0 + 2 ** -8 + 2 ** -20)])
    bits = si._to_bf16_bits(v)
    assert bits.tolist() == [0x3F80, 0x3F82, 0xBF81]


def test_workload_tables():
    assert len(si.workload("router_small")) == 1
    d = si.workload("dotprod")
    assert [c.seed for c in d] == list(range(1, 13))
    assert {(c.K, c.N) for c in d} == {(7168, 256), (7168, 384), (2880, 128)}
    s = si.workload("splitk")
    assert [c.seed for c in s] == list(range(101, 113)) and {c.M for c in s} == {5, 8, 12, 16}
    p = si.workload("projection")
    assert all(c.ly == c.N + 64 for c in p) and len(p) == 15
    e = si.workload("edge")
    assert len(e) == 200
    assert all(1 <= c.M <= 16 and 1 <= c.N <= 1024 and 1 <= c.K <= 8200 and c.N <= c.ly <= c.N + 67
               for c in e)
    assert any(c.K % 8 != 0 for c in e) and any(c.K % 2 == 1 for c in e)
    assert si.edge_cases() == e   # deterministic
    m = si.workload("midm")
    assert len(m) == 18 and all(17 <= c.M <= 64 for c in m) and {c.M for c in m} >= {17, 32, 64}
    assert [c.seed for c in m] == list(range(401, 411)) + list(range(421, 429))
    me = si.workload("midm_edge")
    assert len(me) == 40 and si.midm_edge_cases() == me
    assert all(17 <= c.M <= 64 and c.K % 16 == 0 and 16 <= c.K <= 8192 and c.N <= c.ly <= c.N + 67 for c in me)


def test_embed_rows():
    a = np.arange(6, dtype=np.uint16).reshape(2, 3)
    e = si.embed_rows(a, 5, fill=9)
    assert e.tolist() == [0, 1, 2, 9, 9, 3, 4, 5, 9, 9]


def test_f32_weights_are_seeded_full_precision():
    c = si.Case("f", M=2, N=16, K=300, seed=9)
    a, b = si.make_f32_weights(c), si.make_f32_weights(c)
    assert a.dtype == np.float32 and a.shape == (16, 300) and np.array_equal(a, b)
    assert np.any(a.view(np.uint32) & 0xFFFF)          # not bf16-representable
    assert abs(float(a.std()) - 0.02) < 0.003
