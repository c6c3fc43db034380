"""Host logic of the split tiles (no GPU): the tile lists the forward's down projection
y = h @ W2^T runs in 256 x 512 tiles when the last round of whole tiles would leave CTA
pairs idle.  Every tile's reduction must be covered exactly once, by one whole entry or by
the two pieces of a split tile; the pairs' k-block counts must be even; and each pair's
tail must start with its prefix piece and end with its suffix piece."""
import pytest

from bwd_gemm_epilogue_gb300 import binding as b

MIN_PIECE = 8   # k-blocks: the plan moves boundaries that would cut shorter pieces


def _tiles(M, N):
    return -(-M // 256) * (N // 512)


def _check(M, N, K, units):
    plan = b.swiglu_mlp_split_plan(M, N, K, units)
    assert plan is not None
    kb = -(-K // 64)
    n = _tiles(M, N)
    cover = {t: [] for t in range(n)}
    by_pair = {u: [] for u in range(units)}
    for u, t, k0, k1, sid in plan:
        assert 0 <= u < units and 0 <= t < n and 0 <= k0 < k1 <= kb
        cover[t].append((k0, k1, sid, u))
        by_pair[u].append((t, k0, k1, sid))
    pieces = {}
    for t, entries in cover.items():
        entries.sort()
        if len(entries) == 1:
            k0, k1, sid, _ = entries[0]
            assert (k0, k1, sid) == (0, kb, -1), (t, entries)
        else:
            # a split tile: a prefix [0, r) and a suffix [r, kb) with one split index
            assert len(entries) == 2, (t, entries)
            (a0, a1, sa, ua), (c0, c1, sc, uc) = entries
            assert a0 == 0 and a1 == c0 and c1 == kb and sa == sc >= 0 and ua != uc
            assert MIN_PIECE <= a1 <= kb - MIN_PIECE
            assert abs(ua - uc) == 1       # neighbouring runs share the tile
            pieces[sa] = (t, ua, uc)
    assert sorted(pieces) == list(range(len(pieces)))   # split indices 0..n_split-1, each once
    assert len(pieces) <= 80
    # whole rounds round robin, then even k-block shares
    loads = [sum(k1 - k0 for _, k0, k1, _ in by_pair[u]) for u in range(units)]
    assert max(loads) - min(loads) <= 2 * MIN_PIECE + 1, loads
    whole_rounds = n // units - 1
    for u in range(units):
        head = [t for t, k0, k1, sid in by_pair[u][:whole_rounds]]
        assert head == [u + r * units for r in range(whole_rounds)]
    # every pair's tail starts with its prefix piece (k-block 0, with all other pairs) and
    # ends with its suffix piece
    for u in range(units):
        tail = by_pair[u][whole_rounds:]
        for i, (t, k0, k1, sid) in enumerate(tail):
            if sid >= 0 and k0 == 0:
                assert i == 0, (u, tail)
            elif sid >= 0:
                assert i == len(tail) - 1, (u, tail)
    return plan, pieces


def test_target_down_projection_plan():
    # 308 tiles of 256 x 512 over 76 pairs: 3 whole rounds, then 80 tiles' k-blocks shared
    # (four rounds of whole tiles would leave a fifth round of 4 tiles)
    plan, pieces = _check(11136, 3584, 14336, 76)
    assert len(pieces) > 60
    assert len(plan) == 308 + len(pieces)


@pytest.mark.parametrize("M,N,K,units", [
    (5120, 4096, 6400, 76),      # 160 tiles: 2.1 rounds, 100 k-blocks
    (11136, 3584, 14336, 74),
    (11136, 3584, 14336, 60),
    (8192, 4096, 8192, 76),      # 128 k-blocks
    (6000, 5120, 7168, 71),      # ragged rows, an odd pair count
    (16384, 8192, 16384, 76),    # 512 tiles
])
def test_plans_cover_every_tile_once(M, N, K, units):
    _check(M, N, K, units)


@pytest.mark.parametrize("M,N,K,units", [
    (11136, 3584 + 256, 14336, 76),   # N not a multiple of 512
    (11136, 3584, 4096, 76),          # short reduction: plain 256 x 256 tiles
    (200, 3584, 14336, 76),           # fewer than 256 rows
    (1024, 1024, 14336, 76),          # 8 tiles
    (4096, 4096, 11008, 76),          # prefill: 128 tiles, fewer than two rounds
    (4096, 4096, 11008, 200),         # more pairs than tiles
])
def test_shapes_without_split_tiles(M, N, K, units):
    assert b.swiglu_mlp_split_plan(M, N, K, units) is None


def test_forward_workspace_holds_the_split_sums():
    M, D, H, Dout = 11136, 3584, 14336, 3584
    split = 20480 + 80 * 32 * 32 * 128 * 4
    assert b.swiglu_mlp_fwd_workspace_size(M, D, H, Dout) == M * H * 2 + split
    # no split tiles for these down projections: h alone
    assert b.swiglu_mlp_fwd_workspace_size(M, D, 4096, Dout) == M * 4096 * 2
    assert b.swiglu_mlp_fwd_workspace_size(4096, 4096, 11008, 4096) == 4096 * 11008 * 2
