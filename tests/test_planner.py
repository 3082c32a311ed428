"""The launch planner through the C ABI's planning queries (host only, no GPU): the
split-tail piece count, the CTA-pair / single-CTA choice, the self-chunk split of the
CTA-pair AG tiling and the gather's copy order. The calls run this same code."""
import math

import pytest

from gemm_overlap_gemms_gb300 import _build, ub

PAIRS, SLOTS = 76, 152          # GB300: 152 SMs, 76 CTA pairs


@pytest.fixture(scope="module", autouse=True)
def lib():
    _build.build()
    return ub.load()


def _allowed(tiles, pairs, kb):
    rem = tiles % pairs
    if rem == 0:
        return 1
    return max(1, min(pairs // rem, 8, kb // 16))


@pytest.mark.parametrize("pairs", [1, 3, 37, 76])
@pytest.mark.parametrize("kb", [1, 15, 16, 40, 64, 128, 224, 448, 1000])
def test_tail_split_stays_within_its_limits(pairs, kb):
    for tiles in range(1, 3 * pairs + 2):
        s = ub.plan_tail_split(tiles, pairs, kb)
        w = ub.plan_tail_split(tiles, pairs, kb, widest=True)
        rem = tiles % pairs
        assert 1 <= s <= w == _allowed(tiles, pairs, kb), (tiles, pairs, kb, s, w)
        if rem == 0:
            assert s == 1                       # whole waves: nothing to share
        if s > 1:
            assert rem * s <= pairs             # one piece per idle pair at most
            assert kb // s >= 16                # pieces of at least 16 k-blocks


def test_tail_split_grows_with_k():
    """The fix-up is a fixed time per added piece, so longer tiles afford more pieces."""
    for tiles in (80, 96, 112, 256, 300, 384):
        prev = 1
        for kb in (16, 32, 64, 96, 128, 224, 448, 896):
            s = ub.plan_tail_split(tiles, PAIRS, kb)
            assert s >= prev, (tiles, kb, s, prev)
            prev = s


@pytest.mark.parametrize("what,tiles,kb,gathered,split", [
    # measured on GB300, whole tiles against a split last wave (one call from a CUDA graph,
    # L2 flushed before it, median of 20; bench.py --case ... --streamk 0|n gives the same)
    ("QKV AG T=2048 (one whole wave): 53.8 us whole, 55.8 split in 2, 62.0 in 3", 96, 64, True, False),
    ("SwiGLU fc1 AG+SwiGLU T=1024 (one whole wave): 62.5 us whole, 64.1 split in 2", 112, 64, True, False),
    ("QKV AG T=5120 (three whole waves): 96.1 us whole, 90.5 split in 4", 240, 64, True, True),
    ("SwiGLU fc1 AG+SwiGLU T=3072 (four whole waves): 124.0 us whole, 119.3 split in 2", 336, 64, True, True),
    ("SwiGLU fc2 RS T=512: 78.4 us whole, 57.9 split in 2", 32, 224, False, True),
    ("SwiGLU fc2 RS T=1536: 144.6 us whole, 113.2 split in 3", 96, 224, False, True),
    ("SwiGLU fc2 RS T=4096: 292.6 us whole, 268.8 split in 2", 256, 224, False, True),
    ("large RS K=1024 T=2048: 180.7 us whole, 168.4 split in 2", 256, 128, False, True),
    ("large RS K=3584 T=2048: 614.2 us whole, 561.7 split in 2", 256, 448, False, True),
])
def test_tail_split_follows_the_measured_winner(what, tiles, kb, gathered, split):
    assert (ub.plan_tail_split(tiles, PAIRS, kb, gathered=gathered) > 1) == split, what


def test_gathered_ag_splits_with_no_whole_wave_or_after_two():
    """One whole wave in front: the tail waits for the gather's last rows, no split. No
    whole wave: every tile is split over the idle pairs when the fix-up pays."""
    for tiles in range(1, 6 * PAIRS):
        s = ub.plan_tail_split(tiles, PAIRS, 64, gathered=True)
        if tiles // PAIRS == 1:
            assert s == 1, tiles
        assert s <= ub.plan_tail_split(tiles, PAIRS, 64, widest=True, gathered=True)
    # QKV at T = 256 / 512 (12 / 24 pair tiles, 64 k-blocks): split
    assert ub.plan_tail_split(12, PAIRS, 64, gathered=True) > 1
    assert ub.plan_tail_split(24, PAIRS, 64, gathered=True) > 1
    # QKV at T = 2048 (96 tiles, one whole wave): whole tiles
    assert ub.plan_tail_split(96, PAIRS, 64, gathered=True) == 1


def test_plan_path_respects_forced_options():
    for single, pair_tiles, kb in [(96, 48, 64), (192, 96, 64), (1024, 512, 224), (7, 4, 8)]:
        assert ub.plan_path(single, pair_tiles, kb, SLOTS, PAIRS, cta_pair=0) == (False, False)
        assert ub.plan_path(single, pair_tiles, kb, SLOTS, PAIRS, cta_pair=1, streamk=0) == (True, False)
        assert ub.plan_path(single, pair_tiles, kb, SLOTS, PAIRS, cta_pair=1, streamk=1) == (True, True)


def test_plan_path_cost_model_choices():
    # whole waves of pair tiles: pairs, no split (nothing left to share)
    assert ub.plan_path(2 * 2 * PAIRS, 2 * PAIRS, 224, SLOTS, PAIRS) == (True, False)
    # the SwiGLU fc2 RS at T = 4096 (256 pair tiles, 224 k-blocks): pairs, last wave split
    assert ub.plan_path(512, 256, 224, SLOTS, PAIRS) == (True, True)
    # QKV AG at T = 2048 (96 pair tiles, 64 k-blocks): pairs, whole tiles
    assert ub.plan_path(192, 96, 64, SLOTS, PAIRS, gathered=True) == (True, False)
    # QKV AG at T = 5120 (240 pair tiles): pairs, last wave split
    assert ub.plan_path(480, 240, 64, SLOTS, PAIRS, gathered=True) == (True, True)
    # one wave either way: pairs (a third less L2 traffic per tile)
    assert ub.plan_path(8, 4, 2, SLOTS, PAIRS) == (True, False)
    # AG at T = 512 (N = 7168): 112 chunk-aligned single tiles in one wave against 84
    # pair tiles in two, too short to split (64 k-blocks): single CTAs
    assert ub.plan_path(112, 84, 64, SLOTS, PAIRS) == (False, False)


def _row_tiles(T, c, self_rank, head):
    parts = [head, T - self_rank * c - head, self_rank * c]
    return sum(math.ceil(r / 256) for r in parts if r > 0)


@pytest.mark.parametrize("tp", [1, 2, 4, 8])
@pytest.mark.parametrize("n_tiles", [12, 28])
def test_self_head_split_only_when_it_saves_a_wave(tp, n_tiles):
    for T in list(range(tp * 8, 8193, tp * 52)) + [1140, 1316, 2280, 2956, 8192]:
        T -= T % tp
        c = T // tp
        for self_rank in sorted({0, tp - 1, tp // 2}):
            head = ub.plan_ag_self_head(T, tp, self_rank, n_tiles, PAIRS)
            whole = c // 256 * 256
            assert head in (c, whole), (T, tp, self_rank, head)
            waves = lambda h: math.ceil(_row_tiles(T, c, self_rank, h) * n_tiles / PAIRS)
            if head != c:
                assert waves(head) < waves(c), (T, tp, self_rank)
            elif whole != c:
                assert waves(whole) >= waves(c), (T, tp, self_rank)


def test_self_head_cases():
    # AG + SwiGLU at T = 1140 (28 N tiles): 140 tiles in two waves instead of 168 in three
    assert ub.plan_ag_self_head(1140, 4, 0, 28, PAIRS) == 256
    # QKV at T = 1140 (12 N tiles): one wave either way, the self chunk stays in place
    assert ub.plan_ag_self_head(1140, 4, 0, 12, PAIRS) == 285
    # 256 divides c: nothing to split
    assert ub.plan_ag_self_head(8192, 4, 0, 28, PAIRS) == 2048


@pytest.mark.parametrize("call", [
    lambda: ub.plan_tail_split(0, PAIRS, 64),
    lambda: ub.plan_tail_split(10, 0, 64),
    lambda: ub.plan_tail_split(10, PAIRS, 0),
    lambda: ub.plan_path(0, 1, 1, SLOTS, PAIRS),
    lambda: ub.plan_path(1, 1, 1, 0, PAIRS),
    lambda: ub.plan_ag_self_head(1142, 4, 0, 28, PAIRS),     # T % tp != 0
    lambda: ub.plan_ag_self_head(1140, 4, 4, 28, PAIRS),     # self outside the ring
    lambda: ub.plan_ag_self_head(1140, 9, 0, 28, PAIRS),     # tp above the maximum
    lambda: ub.plan_gather_parts(4, 0, 285, 286),            # head past the chunk
    lambda: ub.plan_gather_parts(4, 4, 285, 256),            # self outside the ring
    lambda: ub.plan_gather_parts(0, 0, 285, 256),
])
def test_planning_queries_reject_bad_arguments(call):
    with pytest.raises(ub.UbError) as ei:
        call()
    assert ei.value.name == "UB_ERR_ARG"


@pytest.mark.parametrize("tp", [1, 2, 3, 4, 8])
def test_gather_parts_cover_every_row_once_and_flag_after_what_the_gemm_reads(tp):
    for c in (1, 100, 255, 256, 257, 285, 570, 2048):
        heads = sorted({c, c // 256 * 256})
        for self_rank in range(tp):
            for head in heads:
                parts = ub.plan_gather_parts(tp, self_rank, c, head)
                rows = {r: [] for r in range(tp)}
                flags = {r: [] for r in range(tp)}
                for i, (r, lo, hi, flag) in enumerate(parts):
                    assert 0 <= lo < hi <= c
                    rows[r].append((lo, hi))
                    if flag:
                        flags[r].append(i)
                for r in range(tp):
                    cover = sorted(rows[r])
                    assert cover[0][0] == 0 and cover[-1][1] == c
                    assert all(a[1] == b[0] for a, b in zip(cover, cover[1:]))   # no gap, no overlap
                    assert len(flags[r]) == 1                                    # one flag per chunk
                # the other chunks in ring order after the self rank
                others = [r for r, *_ in parts if r != self_rank]
                assert others == [(self_rank + q) % tp for q in range(1, tp)]
                fi = flags[self_rank][0]
                if head < c:
                    # the rows the GEMM reads from the buffer go first, flagged
                    assert parts[0] == (self_rank, head, c, True)
                    assert fi == 0
                else:
                    # read wholly in place: copied last, flagged after its last row
                    assert parts[-1] == (self_rank, 0, c, True)


def test_gather_parts_follow_the_planned_self_head():
    # AG + SwiGLU at T = 1140 on 76 pairs: the self chunk's last 29 rows go first
    head = ub.plan_ag_self_head(1140, 4, 0, 28, PAIRS)
    assert ub.plan_gather_parts(4, 0, 285, head)[0] == (0, 256, 285, True)
    # QKV at T = 1140: the self chunk stays in place and is copied last
    head = ub.plan_ag_self_head(1140, 4, 0, 12, PAIRS)
    assert ub.plan_gather_parts(4, 0, 285, head)[-1] == (0, 0, 285, True)


def test_ag_tile_order_groups_follow_the_first_wave():
    """The CTA-pair AG tile order (76 pairs, tp 4): groups of 8 tile rows when the first
    wave reads only the self chunk's in-place rows, else groups of one chunk's tile rows
    (none below two), so that no group starts tiles of chunks late in the ring."""
    # fc1 (28 N tiles): the self chunk's rows fill the first wave from T = 2280 (3 tile rows)
    assert ub.plan_ag_group_m(4640, 4, 0, 28, 76) == 8
    assert ub.plan_ag_group_m(2280, 4, 0, 28, 76) == 8
    # below that, a chunk's tile rows: T = 2048 has 2 per chunk, T = 1140 fewer than 2
    assert ub.plan_ag_group_m(2048, 4, 0, 28, 76) == 2
    assert ub.plan_ag_group_m(1140, 4, 0, 28, 76) == 0
    # 14 N tiles: the self chunk's 5 tile rows are 70 tiles, less than a wave
    assert ub.plan_ag_group_m(4640, 4, 0, 14, 76) == 4
    # QKV (12 N tiles): 4 tile rows per chunk at T = 4096, a whole first wave at 8192
    assert ub.plan_ag_group_m(4096, 4, 0, 12, 76) == 4
    assert ub.plan_ag_group_m(8192, 4, 0, 12, 76) == 8
    # fewer pairs (an SM margin): the same self chunk fills the first wave sooner
    assert ub.plan_ag_group_m(2048, 4, 0, 28, 50) == 8
    with pytest.raises(ub.UbError):
        ub.plan_ag_group_m(1023, 4, 0, 28, 76)
