"""Host logic of the GEMM planning, through the C ABI (no GPU): which kernel
and tiles a bf16 Linear gets, and the CTA-pair kernel's division of its
tiles' k-blocks among the pairs when tiles are shared out along K.

The division must cover every k-block of every output tile exactly once;
the pairs that share a tile must agree on its counter and know their place
in k order (the last to finish sums the pieces in that order); every shared
piece needs a partial slot of its own, below two per pair.  The kernel runs
this same code (host/device), so a mistake here would be a wrong product."""
import itertools

import pytest

from iteration_level_selective_gb300 import _orca as C

SHAPES_13B = [(15360, 5120), (5120, 5120), (20480, 5120), (5120, 20480), (50257, 5120)]
SHAPES_OTHER = [(2304, 768), (768, 3072), (3072, 768), (520, 12288), (1000, 16384), (4000, 10240), (5000, 13440),
                (20000, 4096), (64, 20480), (520, 131072)]
ROWS = [129, 200, 256, 257, 300, 511, 512, 513, 700, 769, 850, 1024, 1100, 2048, 4096]


@pytest.fixture(scope="module")
def lib():
    try:
        return C.lib()
    except RuntimeError as e:
        pytest.skip(str(e))


def check_division(M, N, K, n_pairs, with_split):
    KB = K // 64
    tiles = ((M + 255) // 256) * ((N + 255) // 256)
    covered = {}
    by_tile = {}
    for p in range(n_pairs):
        for seg in C.orca_gemm_pair_segments(M, N, K, n_pairs, with_split, p):
            tile, m, n, kb0, kb1, pieces, mine, counter, slot = seg
            assert 0 <= tile < tiles and 0 <= kb0 < kb1 <= KB, seg
            assert 0 <= m < (M + 255) // 256 and 0 <= n < (N + 255) // 256, seg
            for kb in range(kb0, kb1):
                assert (tile, kb) not in covered, (M, N, K, n_pairs, p, seg)
                covered[(tile, kb)] = p
            by_tile.setdefault(tile, []).append((p, seg))
    assert len(covered) == tiles * KB, (M, N, K, n_pairs)
    tile_mn = {}
    counters, slots = set(), set()
    for tile, segs in by_tile.items():
        pieces = segs[0][1][5]
        assert len(segs) == pieces and all(s[5] == pieces for _, s in segs)
        mn = {(s[1], s[2]) for _, s in segs}
        assert len(mn) == 1
        tile_mn[tile] = mn.pop()
        if pieces == 1:
            assert segs[0][1][7] == -1 and segs[0][1][8] == -1
            continue
        ordered = sorted(segs, key=lambda x: x[1][6])
        assert [s[6] for _, s in ordered] == list(range(pieces))
        # k order: piece i ends where piece i + 1 starts
        for (_, a), (_, b) in zip(ordered, ordered[1:]):
            assert a[4] == b[3], (a, b)
        assert ordered[0][1][3] == 0 and ordered[-1][1][4] == KB
        c = {s[7] for _, s in segs}
        assert len(c) == 1
        c = c.pop()
        assert c not in counters and 0 <= c < n_pairs
        counters.add(c)
        for _, s in segs:
            assert s[8] not in slots and 0 <= s[8] < 2 * n_pairs
            slots.add(s[8])
    # every (row tile, column tile) exactly once
    assert len(set(tile_mn.values())) == tiles


@pytest.mark.parametrize("N,K", SHAPES_13B + SHAPES_OTHER)
def test_pair_division_covers_every_k_block_once(lib, N, K):
    for M in ROWS:
        for n_pairs in (76, 75):
            check_division(M, N, K, n_pairs, True)


@pytest.mark.parametrize("n_pairs", [1, 2, 3, 7, 40, 96])
def test_pair_division_other_pair_counts(lib, n_pairs):
    for (N, K), M in itertools.product([(5120, 20480), (20480, 5120), (1000, 16384), (520, 12288)], [200, 513, 1024]):
        check_division(M, N, K, n_pairs, True)
        check_division(M, N, K, n_pairs, False)


def test_pair_division_without_split_is_whole_tiles(lib):
    for M, (N, K) in itertools.product([200, 1024, 24373], SHAPES_13B):
        for p in (0, 37, 75):
            for seg in C.orca_gemm_pair_segments(M, N, K, 76, False, p):
                assert seg[3] == 0 and seg[4] == K // 64 and seg[5] == 1


def test_pair_division_shares_where_whole_tiles_idle_pairs(lib):
    # the 13B FC1 at 200 rows: 80 tiles on 76 pairs -> 76 stream ranges of 84-85 k-blocks, two pieces a
    # shared tile; the FC2: 20 tiles of 320 k-blocks -> three equal ranges per tile on 60 pairs
    fc1 = [C.orca_gemm_pair_segments(200, 20480, 5120, 76, True, p) for p in range(76)]
    assert {sum(s[4] - s[3] for s in segs) for segs in fc1} <= {84, 85}
    assert max(s[5] for segs in fc1 for s in segs) == 2
    fc2 = [C.orca_gemm_pair_segments(200, 5120, 20480, 76, True, p) for p in range(76)]
    assert [len(s) for s in fc2] == [1] * 60 + [0] * 16
    assert {s[0][4] - s[0][3] for s in fc2[:60]} == {107, 106} and {s[0][5] for s in fc2[:60]} == {3}


# which kernel the 13B and GPT-2-small Linears get on 152 SMs (the engine's scratch given): the
# choices the GB300 measurements behind the planner picked as the faster ones
PLANS = [
    # (M, N, K) -> kernel, tile_n, k_split
    ((24373, 15360, 5120), 2, 256, 0), ((24373, 5120, 20480), 2, 256, 0), ((24373, 20480, 5120), 2, 256, 0),
    ((200, 15360, 5120), 2, 256, 0), ((200, 5120, 5120), 0, 128, 0), ((200, 20480, 5120), 2, 256, 2),
    ((200, 5120, 20480), 2, 256, 1), ((300, 20480, 5120), 0, 256, 0), ((600, 15360, 5120), 0, 256, 0),
    ((600, 5120, 5120), 2, 256, 0), ((700, 5120, 20480), 2, 256, 0), ((1024, 5120, 20480), 2, 256, 2),
    ((64, 768, 3072), 1, 64, 0), ((64, 2304, 768), 0, 32, 0), ((600, 2304, 768), 0, 128, 0),
]


@pytest.mark.parametrize("shape,kernel,tile_n,k_split", PLANS)
def test_plan_choices(lib, shape, kernel, tile_n, k_split):
    r = C.orca_gemm_plan_query(*shape, 152)
    assert (r["kernel"], r["tile_n"], r["k_split"]) == (kernel, tile_n, k_split), r
    assert 0 <= r["code"] < 64
    assert (r["code"] in (40, 41)) == (kernel == 2) and (r["code"] == 41) == (k_split > 0)


def test_plan_without_scratch_never_shares_tiles(lib):
    for M, (N, K) in itertools.product(ROWS, SHAPES_13B + SHAPES_OTHER):
        r = C.orca_gemm_plan_query(M, N, K, 152, with_scratch=False)
        assert r["k_split"] == 0


def test_plan_and_segments_reject_bad_arguments(lib):
    for args in [(0, 128, 64, 152), (64, 0, 64, 152), (64, 128, 100, 152), (64, 128, 64, 1)]:
        with pytest.raises(C.OrcaError):
            C.orca_gemm_plan_query(*args)
    for args in [(64, 128, 100, 76, True, 0), (64, 128, 64, 0, True, 0), (64, 128, 64, 76, True, 76),
                 (64, 128, 64, 76, True, -1)]:
        with pytest.raises(C.OrcaError):
            C.orca_gemm_pair_segments(*args)
