"""Host-side restatements of what the kernels derive from a plan (no GPU)."""
import latency_skinny_bf16_gb300 as sk


def check_tc_geometry(p, M, N, K):
    """What the tcgen05 kernel derives from a plan, restated: W rows in groups
    of 8, grid_y balanced ranges of groups, tiles of at most block_n rows (one
    tile per CTA when K is split over a cluster), K slices of whole ring
    stages, and a ring (per stage: VP W rows and the MT token rows of X, 128
    bytes each per 64-element box) that fits the shared memory asked for and
    can receive the cluster's partial sums."""
    tm, s, bk, C = p["block_n"], p["split_k"], p["stage_k"], p["grid_y"]
    G = -(-N // 8)
    assert p["backend"] == sk.SKINNY_BACKEND_TCGEN05 and p["consumer"] == sk.SKINNY_CONSUMER_MMA
    assert tm in (64, 128) and s in (1, 2, 4, 8) and p["grid_x"] == s and p["threads"] == 192
    assert 1 <= C <= G
    ranges = [(c * G // C, (c + 1) * G // C) for c in range(C)]
    assert ranges[0][0] == 0 and ranges[-1][1] == G and all(a < b for a, b in ranges)
    assert all(ranges[i][1] == ranges[i + 1][0] for i in range(C - 1))
    gmax = max(b - a for a, b in ranges)
    assert gmax - min(b - a for a, b in ranges) <= 1            # balanced to one group
    T = -(-gmax // (tm // 8))
    vg = -(-gmax // T)
    assert 8 * vg <= tm
    if s > 1:
        assert T == 1
    assert bk % 64 == 0 and 64 <= bk <= 256
    assert p["k_chunk"] % bk == 0 and s * p["k_chunk"] >= K      # trailing ranks may be empty (they add 0)
    mt = 16 if M <= 16 else 32 if M <= 32 else 64
    ring = p["stages"] * (bk // 64) * (8 * vg + mt) * 128
    # 256 tensor-memory columns per CTA (four sets of 64 / mt accumulators of mt
    # columns): the shared memory asked for caps the CTAs per SM at two
    assert 77 * 1024 <= p["smem_bytes"] <= 227 * 1024
    assert (228 * 1024 // p["smem_bytes"]) * 256 <= 512
    assert ring + 8 * (2 * p["stages"] + 9) + 16 + 1024 <= p["smem_bytes"]
    if s > 1:
        assert ring >= s * M * (-(-8 * vg // s)) * 4            # S slots of M x ceil(VP / S) fp32
    return G, C, vg
