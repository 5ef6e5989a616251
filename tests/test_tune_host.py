"""Host logic of the tuning sweep: candidate lists and merging of winners into table lines."""
import pytest

tune = pytest.importorskip("latency_skinny_bf16_gb300.tune")


def test_candidates_cover_both_backends_and_respect_k16():
    c = tune.candidates(8, 7168)
    assert {x["backend"] for x in c} == {1, 2}
    assert any(x["backend"] == 2 and x["consumer"] == 2 for x in c)
    c = tune.candidates(8, 7176)     # K % 16 != 0: no MMA consumer
    assert not any(x["backend"] == 2 and x["consumer"] == 2 for x in c)


def test_merge_rows_merges_consecutive_equal_winners():
    a = dict(backend=2, consumer=2, split_k=8, stages=4, block_n=0)
    b = dict(backend=1, consumer=0, split_k=0, stages=0, block_n=1)
    rows = [(1, b, 3.0), (2, a, 3.5), (3, a, 3.6), (4, a, 3.7), (5, b, 4.0), (7, a, 4.1)]
    lines = tune.merge_rows(7168, 256, rows)
    # ranges cover 1..16: a gap (M=6 not tuned) goes to the line before it
    assert [(l[2], l[3], l[4]) for l in lines] == [(1, 1, 1), (2, 4, 2), (5, 6, 1), (7, 16, 2)]
    assert lines[1][10] == [3.5, 3.6, 3.7]


def test_merge_rows_never_crosses_the_8_token_boundary():
    a = dict(backend=2, consumer=2, split_k=1, stages=0, block_n=0)
    rows = [(3, a, 8.7), (8, a, 9.1), (12, a, 13.0), (16, a, 13.6)]
    lines = tune.merge_rows(7168, 2112, rows)
    assert [(l[2], l[3]) for l in lines] == [(3, 8), (12, 16)]   # M 9..11 left to the default rule
