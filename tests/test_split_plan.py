"""Host-side checks of the ws entry point's split plan (no GPU): the plan and
items come from the library's own code (nf4_split_plan / nf4_split_item).

Invariants: every stage of every tile is run by exactly one pair; whole waves
stay whole; a split tile is finished by the pair holding its stage 0, as that
pair's last item, and the partners it adds are exactly the other pairs that
hold stages of the tile, each of which runs that part right after its whole
tiles (every pair has the same number of those, so the part is written before
the finishing pair, which runs its part last, needs it) and writes at most one
partial.
"""
from __future__ import annotations

import itertools

import pytest

import backward_gemm_gb300 as nb


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from backward_gemm_gb300.build import build

    build()
    nb.lib()


CASES = [(48, 24, 76), (96, 140, 76), (560, 24, 76), (512, 224, 76), (6, 3, 76), (6, 1, 76),
         (1, 24, 76), (75, 50, 76), (77, 45, 76), (20, 140, 76), (7, 200, 3), (5, 700, 4),
         (3, 1000, 74), (1792, 64, 76), (65, 170, 64), (2, 200, 2), (152, 24, 76), (10, 90, 8),
         (4, 64, 76), (80, 9, 76)]


@pytest.mark.parametrize("T,S,P", CASES)
def test_split_plan_covers_every_stage_once(T, S, P):
    dp, sk = nb.split_plan(T, S, P)
    assert dp + sk == T
    if sk:
        assert dp % P == 0 and sk == T % P and S * (P - sk) >= 40 * P
    else:
        assert T % P == 0 or S * (P - T % P) < 40 * P or S <= 1 or P <= 1
    seen = {}
    items = {p: nb.split_items(T, S, P, p) for p in range(P)}
    for p, its in items.items():
        for (t, s0, s1, q0, q1) in its:
            assert 0 <= t < T and 0 <= s0 < s1 <= S
            for s in range(s0, s1):
                assert (t, s) not in seen, (t, s, p, seen.get((t, s)))
                seen[(t, s)] = p
    assert len(seen) == T * S
    # whole tiles round-robin in the first part
    for t in range(dp):
        assert all(seen[(t, s)] == t % P for s in range(S))


@pytest.mark.parametrize("T,S,P", CASES)
def test_split_tiles_finish_after_their_partials(T, S, P):
    dp, _ = nb.split_plan(T, S, P)
    items = {p: nb.split_items(T, S, P, p) for p in range(P)}
    owners = {}
    for p, its in items.items():
        for k, (t, s0, s1, q0, q1) in enumerate(its):
            owners.setdefault(t, []).append((s0, p, k))
    partial_writes = {p: 0 for p in range(P)}
    for p, its in items.items():
        for k, (t, s0, s1, q0, q1) in enumerate(its):
            parts = sorted(owners[t])
            if len(parts) == 1:
                assert (s0, s1) == (0, S) and q1 < q0
                continue
            if s0 == 0:
                # finishing pair: last item of its run; partners = the others, in order
                assert k == len(its) - 1
                busy = [q for q in range(q0, q1 + 1) if any(it[0] >= dp for it in items[q])]
                assert [pp for _, pp, _ in parts[1:]] == busy
                assert q0 == p + 1
            else:
                assert q1 < q0
                ndp = sum(1 for it in its if it[0] < dp)
                assert k == ndp, "a partial part is its pair's first item after its whole tiles"
                partial_writes[p] += 1
    assert max(partial_writes.values()) <= 1


def test_split_plan_rejects_bad_arguments():
    with pytest.raises(ValueError):
        nb.split_plan(0, 4, 76)
    with pytest.raises(ValueError):
        nb.split_items(4, 4, 76, 76)


def test_tile_rows_choice_for_the_workloads():
    """512-token tiles need >= 8 stages and >= pairs / 2 tiles: q_proj (24 such
    tiles for 76 pairs) and N = 256 (4 stages) keep 256."""
    P = 76
    assert nb.tile_rows(2048, 1536, 1536, P) == 256          # q_proj
    assert nb.tile_rows(4096, 256, 1536, P) == 256           # k_proj / v_proj
    assert nb.tile_rows(4096, 8960, 1536, P) == 512          # up_proj
    assert nb.tile_rows(4096, 1536, 8960, P) == 512          # down_proj
    assert nb.tile_rows(8191, 4096, 14336, P) == 512         # large_b
    assert nb.tile_rows(8191, 14336, 4096, P) == 512         # large_a
    assert nb.tile_rows(256, 4096, 4096, P) == 256           # one 256-token block
    assert nb.tile_rows(4096, 448, 4096, P) == 256           # 7 stages
    assert nb.tile_rows(4096, 512, 4096, P) == 512           # 8 stages
    with pytest.raises(ValueError):
        nb.tile_rows(0, 64, 64, P)


def test_backward_b_token_splits():
    """GemmBackwardB cuts the token range (the contraction, 64 tokens a stage)
    only when its (256 x 256) output tiles leave pairs idle, into at most
    pairs // tiles runs of at least 8 stages each."""
    L = nb.lib()
    P = 76
    for M, K, N in [(4096, 1536, 1536), (4096, 16, 8960), (4096, 16, 1536), (512, 16, 256),
                    (511, 16, 256), (64, 8, 8), (100000, 16, 256), (4096, 4096, 14336)]:
        tiles = -(-K // 256) * -(-N // 256)
        stages = -(-M // 64)
        s = int(L.nf4_gemm_backward_b_splits(M, K, N, P))
        assert s >= 1
        if tiles >= P:
            assert s == 1, (M, K, N)
        else:
            assert s * tiles <= P and (s == 1 or 8 * s <= stages), (M, K, N, s)
            assert s == max(1, min(P // tiles, stages // 8)), (M, K, N, s)
    assert int(L.nf4_gemm_backward_b_splits(4096, 16, 8960, P)) == 2     # rank-16 adapter, 35 tiles
    assert int(L.nf4_gemm_backward_b_splits(4096, 1536, 1536, P)) == 2   # 36 tiles
    assert int(L.nf4_gemm_backward_b_splits(511, 16, 256, P)) == 1       # 8 stages: one run
    assert int(L.nf4_gemm_backward_b_splits(0, 16, 256, P)) == 1         # no tokens
    for bad in [(-1, 16, 256, P), (64, 0, 256, P), (64, 16, 0, P), (64, 16, 256, 0)]:
        assert int(L.nf4_gemm_backward_b_splits(*bad)) == -1
