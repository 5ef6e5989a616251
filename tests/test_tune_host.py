"""Host logic of the tuning sweep: candidate lists and merging of winners into table lines."""
import pytest

tune = pytest.importorskip("latency_skinny_bf16_gb300.tune")


def test_candidates_cover_both_backends_and_respect_k16():
    c = tune.candidates(8, 7168)
    assert {x["backend"] for x in c} == {1, 2, 4}
    assert {x["backend"] for x in tune.candidates(3, 7168)} == {1, 2}
    assert any(x["backend"] == 2 and x["consumer"] == 2 for x in c)
    c = tune.candidates(8, 7176)     # K % 16 != 0: no MMA consumer
    assert not any(x["backend"] == 2 and x["consumer"] == 2 for x in c)


def test_merge_rows_merges_consecutive_equal_winners():
    a = dict(backend=2, consumer=2, split_k=8, stages=4, block_n=0)
    b = dict(backend=1, consumer=0, split_k=0, stages=0, block_n=1)
    rows = [(1, b, 3.0), (2, a, 3.5), (3, a, 3.6), (4, a, 3.7), (5, b, 4.0), (7, a, 4.1)]
    lines = tune.merge_rows(7168, 256, rows)
    # a gap (M=6 not tuned) goes to the line before it; the last line ends with its token bucket
    assert [(l[2], l[3], l[4]) for l in lines] == [(1, 1, 1), (2, 4, 2), (5, 6, 1), (7, 8, 2)]
    assert lines[1][10] == 0 and lines[1][11] == [3.5, 3.6, 3.7]     # clusters: the planner's own


def test_tc_candidates_span_cluster_sizes_and_tile_heights():
    c = tune.tc_candidates(16, 7168, 2112, num_sms=152)
    assert {x["split_k"] for x in c} == {1, 2, 4, 8}
    assert all(x["backend"] == 4 and x["stage_k"] in (128, 256) for x in c)
    # row-range counts: the planner's (0) and those giving 6..16 groups of 8 rows per tile
    # that fit one wave (clusters of 8: 34 at most)
    assert {x["clusters"] for x in c if x["split_k"] == 8} == {0, 17, 22, 33}
    assert all(x["clusters"] * x["split_k"] <= 2 * 152 for x in c)
    assert {x["split_k"] for x in tune.tc_candidates(16, 512, 256)} == {1, 2}   # K < 2 * S * 128 refused


def test_merge_rows_never_crosses_the_8_token_boundary():
    a = dict(backend=2, consumer=2, split_k=1, stages=0, block_n=0)
    rows = [(3, a, 8.7), (8, a, 9.1), (12, a, 13.0), (16, a, 13.6)]
    lines = tune.merge_rows(7168, 2112, rows)
    assert [(l[2], l[3]) for l in lines] == [(3, 8), (12, 16)]   # M 9..11 left to the default rule


def test_mid_m_candidates_are_tensor_core_only():
    c = tune.candidates(17, 7168, 256)
    assert c and all((x["backend"], x["consumer"]) in ((2, 2), (4, 0)) for x in c)
    assert {x["backend"] for x in c} == {2, 4}
    c = tune.candidates(40, 7176, 256)      # K % 16 != 0: only the tcgen05 backend (any K)
    assert c and all(x["backend"] == 4 for x in c)
    # large weights: tcgen05 plans at every M
    assert any(x["backend"] == 4 for x in tune.candidates(1, 1536, 24576))
    assert not any(x["backend"] == 4 for x in tune.candidates(4, 7168, 256))   # tiny M on small weights
    assert any(x["backend"] == 4 for x in tune.candidates(12, 7168, 256))
    assert [tune.token_bucket(m) for m in (1, 8, 9, 16, 17, 32, 33, 64)] == [8, 8, 16, 16, 32, 32, 64, 64]


def test_merge_rows_respects_every_token_bucket():
    a = dict(backend=2, consumer=2, split_k=8, stages=0, block_n=0, stage_k=0)
    rows = [(12, a, 5.0), (16, a, 5.1), (17, a, 6.0), (24, a, 6.1), (32, a, 6.3), (40, a, 7.0), (64, a, 8.0)]
    lines = tune.merge_rows(7168, 256, rows)
    assert [(l[2], l[3]) for l in lines] == [(12, 16), (17, 32), (40, 64)]   # 33..39 left to the default
    # a shape whose 33..64 bucket does not run ends its last line at 32
    lines = tune.merge_rows(14336, 7168, rows[:5])
    assert [(l[2], l[3]) for l in lines] == [(12, 16), (17, 32)]


def test_install_replaces_the_lines_of_tuned_shapes(tmp_path):
    path = tmp_path / "table.inc"
    path.write_text("// header\n{7168, 256, 1, 2, 1, 0, 0, 1, 0, 0},  // a\n"
                    "{1536, 24576, 1, 8, 1, 2, 0, 64, 0, 0},  // b\n{1536, 24576, 9, 16, 2, 2, 1, 0, 0, 0},  // c\n"
                    "{7168, 384, 1, 1, 1, 0, 0, 1, 0, 0},  // d\n")
    new = ["{1536, 24576, 1, 16, 4, 0, 1, 0, 0, 128},  // e"]
    tune.install(new, str(path))
    lines = path.read_text().strip().split("\n")
    assert lines == ["// header", "{7168, 256, 1, 2, 1, 0, 0, 1, 0, 0},  // a", new[0],
                     "{7168, 384, 1, 1, 1, 0, 0, 1, 0, 0},  // d"]
    tune.install(["{2880, 128, 1, 3, 1, 0, 0, 2, 0, 0},  // f"], str(path))   # a new shape goes at the end
    assert path.read_text().strip().split("\n")[-1].endswith("// f")
    # a shape tuned over part of its M range keeps its lines outside that range:
    # the new line meets no old one, so it goes at the end
    tune.install(["{7168, 256, 17, 32, 4, 0, 8, 0, 0, 128, 34},  // g"], str(path))
    lines = path.read_text().strip().split("\n")
    assert "{7168, 256, 1, 2, 1, 0, 0, 1, 0, 0},  // a" in lines and lines[-1].endswith("// g")
    # re-tuning M = 2..32 drops every line it meets: 1..2 and 17..32
    tune.install(["{7168, 256, 2, 32, 2, 2, 4, 0, 0, 0, 0},  // h"], str(path))
    lines = path.read_text().strip().split("\n")
    assert not any(l.endswith("// a") or l.endswith("// g") for l in lines)
    assert sum(l.endswith("// h") for l in lines) == 1


def test_candidates_include_cluster_split_dot_product():
    c = tune.candidates(16, 7168, 256)
    splits = {(x["split_k"], x["block_n"]) for x in c if x["backend"] == 1 and x["consumer"] == 2}
    assert {(2, 16), (4, 16), (8, 32)} <= splits
    assert not any(x["backend"] == 1 and x["split_k"] > 1 for x in tune.candidates(16, 7176, 256))   # K % 32


def test_fill_gaps_extends_the_next_line_down():
    sk = pytest.importorskip("latency_skinny_bf16_gb300")
    a = dict(backend=2, consumer=2, split_k=1, block_n=0, stages=0, stage_k=1024, clusters=0)
    b = dict(backend=2, consumer=2, split_k=2, block_n=0, stages=0, stage_k=0, clusters=0)
    # 2112 x 7168: the first plan stops planning at M = 11 (its X slice); the second takes 11
    out = tune.fill_gaps(7168, 2112, [(9, 10, a), (12, 15, b)], 152)
    assert [(lo, hi) for lo, hi, _ in out] == [(9, 10), (11, 15)]
    # no gap across a token bucket (8 -> 9): left for the default rule of the bucket
    out = tune.fill_gaps(7168, 2112, [(2, 6, b), (9, 16, b)], 152)
    assert [(lo, hi) for lo, hi, _ in out] == [(2, 6), (9, 16)]
