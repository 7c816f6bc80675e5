"""Pins for the schedule oracle against what the pages print and what the mathematics fixes.

Each pin checks the oracle against something other than itself: the printed wave table and
schedule report ("Split-K and Stream-K: The Last Wave of a GEMM", Cases 1 and 2), the toy
4-SM case of its Mental model figure, the Triton driver's printed partition (Case 3), and
brute force over small shapes (every (tile, k) iteration covered exactly once, balanced
units, the owner being the lowest contributor).
"""
import csv
import itertools
import os

import pytest

from oracle import schedule as S


def _rows(path, delimiter=","):
    with open(path) as f:
        return [r for r in csv.reader((l for l in f if not l.startswith("#")), delimiter=delimiter)]


def test_wave_table(golden_dir):
    rows = _rows(os.path.join(golden_dir, "wave_table.csv"))
    assert len(rows) == 15
    for m, n, sms, tiles, w, tail, util in rows:
        t, ww, tl, u = S.waves(int(m), int(n), int(sms))
        assert (t, ww, tl) == (int(tiles), int(w), int(tail))
        assert f"{100 * u:.1f}" == util


def test_thesis_example():
    # 144 tiles on a 132-SM part: the second wave keeps 12 SMs busy, 54.5% overall.
    tiles, w, tail, util = S.waves(1536, 1536, 132)
    assert (tiles, w, tail) == (144, 2, 12)
    assert round(100 * util, 1) == 54.5


def test_schedule_report(golden_dir):
    rows = _rows(os.path.join(golden_dir, "schedule_sim.psv"), delimiter="|")
    assert len(rows) == 20
    by_shape = {}
    for r in rows:
        by_shape.setdefault(tuple(int(x) for x in r[:4]), []).append(r)
    for (m, n, k, sms), expect in by_shape.items():
        tiles, iters, ideal, got = S.report_rows(m, n, k, sms)
        assert (tiles, iters) == (int(expect[0][4]), int(expect[0][5]))
        assert f"{ideal:.1f}" == expect[0][6]
        assert len(got) == len(expect) == 5
        for (name, t, eff), e in zip(got, expect):
            assert name == e[7]
            assert f"{t:.1f}" == e[8], (m, n, k, name)
            assert f"{100 * eff:.1f}" == e[9]


def test_toy_case(golden_dir):
    # Mental model: 4 SMs, 5 tiles x 4 iterations (M=128, N=640, K=256), forced to 4 units.
    dp = S.build_plan(128, 640, 256, 4, S.DP)
    assert (dp.tiles, dp.iters) == (5, 4)
    t = S.makespan(dp, EPI=0, PART=0)
    assert t == 8
    assert 20 / (t * 4) == 0.625
    sk = S.build_plan(128, 640, 256, 4, S.STREAMK)
    per_unit = [sum(s.k_end - s.k_begin for s in segs) for segs in sk.units]
    assert per_unit == [5, 5, 5, 5]
    assert S.makespan(sk, EPI=0, PART=0) == 5
    expect = _rows(os.path.join(golden_dir, "toy_streamk_map.csv"))
    roles = {"FULL": S.FULL, "OWNER": S.OWNER, "PRODUCER": S.PRODUCER}
    got = [(s.unit, s.tile, s.k_begin, s.k_end, s.role) for s in sk.segments()]
    assert got == [(int(u), int(t), int(a), int(b), roles[r]) for u, t, a, b, r in expect]
    # Units 1..3 start with the partial they hand off; the k=0 holder owns the fixup.
    assert [segs[0].role for segs in sk.units] == [S.FULL, S.PRODUCER, S.PRODUCER, S.PRODUCER]
    assert [o for o, _ in S.tile_rows(sk)] == [0, 0, 1, 2, 3]
    # Same toy through the units override rather than the SM count.
    sk2 = S.build_plan(128, 640, 256, 148, S.STREAMK, units=4)
    assert S.plan_map(sk2) == S.plan_map(sk)


def test_streamk_groups_toy(golden_dir):
    # Hand-worked map of the toy case cut into two groups (fixture comment has the steps).
    p = S.build_plan(128, 640, 256, 4, S.STREAMK, sk_groups=2)
    assert p.sk_groups == 2
    expect = _rows(os.path.join(golden_dir, "toy_streamk_groups2_map.csv"))
    roles = {"FULL": S.FULL, "OWNER": S.OWNER, "PRODUCER": S.PRODUCER}
    got = [(s.unit, s.tile, s.k_begin, s.k_end, s.role) for s in p.segments()]
    assert got == [(int(u), int(t), int(a), int(b), roles[r]) for u, t, a, b, r in expect]
    own = [s for s in p.segments() if s.role == S.OWNER][0]
    assert (own.peer_begin, own.n_peers) == (1, 1)
    # One group (0 or 1) is the page's plan.
    for g in (0, 1):
        assert S.plan_map(S.build_plan(128, 640, 256, 4, S.STREAMK, sk_groups=g))[S.HEADER_LEN:] == \
            S.plan_map(S.build_plan(128, 640, 256, 4, S.STREAMK))[S.HEADER_LEN:]


def test_streamk_group_count():
    # "Up to" the requested count: never more groups than tiles or units, and never a group
    # with more units than k-iterations (no empty unit).
    assert S.sk_group_count(5, 4, 4, 8) == 4          # min(8, 5 tiles, 4 units)
    assert S.sk_group_count(16, 1024, 148, 8) == 8
    assert S.sk_group_count(2, 64, 128, 8) == 2         # 64 units on 64 iterations each
    assert S.sk_group_count(2, 64, 129, 8) == 1         # 65 units on a 64-iteration tile: one group
    # 3 tiles x 2 iterations on 6 units: 2 groups would give tiles 2, 1 and units 3, 3, and
    # group 1 would hold 2 iterations for 3 units; so one group.
    assert S.sk_group_count(3, 2, 6, 2) == 1
    assert S.sk_group_count(10, 4, 7, 0) == 1 and S.sk_group_count(10, 4, 7, 1) == 1


def test_streamk_groups_bruteforce():
    # Every grouping: (tile, k) covered exactly once, each unit's range inside one group's
    # tiles, no empty unit, units of a group within one iteration of each other, tiles of
    # different groups never shared, owner = lowest contributor.
    for tiles, iters, units, req in itertools.product(range(1, 13), (1, 2, 3, 4, 8), range(1, 15), (2, 3, 4, 8)):
        if units > tiles * iters:
            continue
        g = S.sk_group_count(tiles, iters, units, req)
        b = S.group_bounds(tiles, iters, units, g)
        assert b[0][0] == 0 and b[-1][1] == tiles * iters
        assert all(b[i][1] == b[i + 1][0] for i in range(units - 1))
        assert all(e > s for s, e in b)
        tg, ug = S.divmod_bounds(tiles, g), S.divmod_bounds(units, g)
        for (t0, t1), (u0, u1) in zip(tg, ug):
            sizes = [b[u][1] - b[u][0] for u in range(u0, u1)]
            assert max(sizes) - min(sizes) <= 1
            assert b[u0][0] == t0 * iters and b[u1 - 1][1] == t1 * iters
        segs = [x for segs in S._streamk_region(0, tiles, iters, units, False, g) for x in segs]
        cover = sorted((x.tile, k) for x in segs for k in range(x.k_begin, x.k_end))
        assert cover == [(t, k) for t in range(tiles) for k in range(iters)]
        for x in segs:
            if x.role == S.OWNER:
                assert all(y.unit > x.unit for y in segs if y.tile == x.tile and y is not x)
                assert x.n_peers == sum(1 for y in segs if y.tile == x.tile) - 1


def test_triton_partition(golden_dir):
    for units, tiles, ipt, total, q, peers in _rows(os.path.join(golden_dir, "triton_partition.csv")):
        units, ipt, total = int(units), int(ipt), int(total)
        assert int(tiles) * ipt == total
        b = S.cdiv_bounds(total, units)
        assert b[0][1] - b[0][0] == int(q)
        if peers:
            most = 0
            for t in range(int(tiles)):
                lo, hi = t * ipt, (t + 1) * ipt
                most = max(most, sum(1 for (x, y) in b if x < hi and y > lo))
            assert most == int(peers)


def test_docc_floor_partition_worked_example():
    # docc StreamK rewrite: block b walks iterations [b*TOTAL/NBLOCKS, (b+1)*TOTAL/NBLOCKS)
    # with integer (floor) division. Worked by hand for TOTAL = 20, NBLOCKS = 6:
    # 0, 20/6 = 3, 40/6 = 6, 60/6 = 10, 80/6 = 13, 100/6 = 16, 120/6 = 20.
    assert S.floor_bounds(20, 6) == [(0, 3), (3, 6), (6, 10), (10, 13), (13, 16), (16, 20)]
    # TOTAL = 7, NBLOCKS = 3: 0, 7/3 = 2, 14/3 = 4, 21/3 = 7.
    assert S.floor_bounds(7, 3) == [(0, 2), (2, 4), (4, 7)]
    # More blocks than iterations leaves some blocks empty: floor(b*2/5) = 0, 0, 0, 1, 1, 2.
    assert S.floor_bounds(2, 5) == [(0, 0), (0, 0), (0, 1), (1, 1), (1, 2)]


def test_docc_floor_partition_aligned_split():
    # docc, aligned split: with NBLOCKS = tiles * S and S dividing the panel count P, block
    # bid owns panels [s*P/S, (s+1)*P/S) of tile t = bid / S (s = bid % S). In the flattened
    # (tile, panel) space that is [t*P + s*P/S, t*P + (s+1)*P/S).
    for tiles in (1, 2, 5, 16):
        for P in (4, 8, 12, 64):
            for Sd in (1, 2, 4):
                if P % Sd:
                    continue
                got = S.floor_bounds(tiles * P, tiles * Sd)
                want = [(bid // Sd * P + bid % Sd * P // Sd, bid // Sd * P + (bid % Sd + 1) * P // Sd)
                        for bid in range(tiles * Sd)]
                assert got == want


def test_docc_floor_partition_invariants():
    # The ranges tile [0, TOTAL) in order, and every size is floor or ceil of TOTAL / NBLOCKS.
    for total in range(0, 60):
        for n in range(1, 25):
            b = S.floor_bounds(total, n)
            assert b[0][0] == 0 and b[-1][1] == total
            assert all(b[i][1] == b[i + 1][0] for i in range(n - 1))
            assert {y - x for x, y in b} <= {total // n, -(-total // n)}


def test_calculate_split_k_worked_examples():
    # The CUTLASS page's Split-K factor heuristic, worked by hand on 148 SMs (2 x 148 = 296
    # tiles switch the split off; the target is 4 x 148 = 592 blocks):
    #   4096 x 4096: 32 x 32 = 1024 tiles >= 296            -> 1
    #   2432 x 2432: 19 x 19 = 361 tiles >= 296             -> 1
    #   2048 x 2048: 16 x 16 = 256 tiles, 592 / 256 = 2.3   -> 3
    #   1024 x 1024: 8 x 8 = 64 tiles, 592 / 64 = 9.25      -> 10
    #   512 x 512: 16 tiles, 592 / 16 = 37                  -> capped at 32
    #   200 x 1000: floor: 1 x 7 = 7 tiles, 592 / 7 = 84.6  -> 32
    #   96 x 512: no whole tile, read as one tile           -> 32
    #   2048 x 2432 on 132 SMs: 16 x 19 = 304 >= 264        -> 1
    #   1536 x 1536 on 132 SMs: 144 tiles, 528 / 144 = 3.67 -> 4
    cases = [((4096, 4096, 148), 1), ((2432, 2432, 148), 1), ((2048, 2048, 148), 3), ((1024, 1024, 148), 10),
             ((512, 512, 148), 32), ((200, 1000, 148), 32), ((96, 512, 148), 32), ((2048, 2432, 132), 1),
             ((1536, 1536, 132), 4)]
    for (m, n, sms), want in cases:
        assert S.calculate_split_k(m, n, 4096, sms) == want, (m, n, sms)
    # K does not enter.
    assert S.calculate_split_k(1024, 1024, 64, 148) == S.calculate_split_k(1024, 1024, 65536, 148)
    with pytest.raises(ValueError):
        S.calculate_split_k(0, 128, 128, 148)


def test_calculate_split_k_invariants():
    # For every shape: a factor in 1..32; 1 exactly when the whole tiles fill two waves;
    # otherwise the factor times the tiles reaches four blocks per SM unless capped, and one
    # split fewer would not; and the factor never grows with M or N.
    for sms in (4, 16, 132, 148, 152):
        prev_row = None
        for m in range(0, 4097, 128):
            row = []
            for n in range(0, 4097, 128):
                mm, nn = max(m, 1), max(n, 1)
                s = S.calculate_split_k(mm, nn, 4096, sms)
                tiles = max(1, (mm // 128) * (nn // 128))
                assert 1 <= s <= 32
                assert (s == 1) == (tiles >= 2 * sms)
                if tiles < 2 * sms and s < 32:
                    assert s * tiles >= 4 * sms and (s - 1) * tiles < 4 * sms
                if row:
                    assert s <= row[-1]
                row.append(s)
            if prev_row:
                assert all(a <= b for a, b in zip(row, prev_row))
            prev_row = row


def test_heuristic_decisions():
    # Case 2 narrative: 2 x 12 < 132 -> all 144 tiles to 132 Stream-K units; on B200
    # (148 SMs, 900 tiles) data-parallel runs 5 full waves and Stream-K takes the 160
    # tiles after them; a tail of 100 on 132 SMs stays data-parallel.
    assert S.heuristic(144, 64, 132) == (S.LABEL_STREAMK, 144, 132, 0)
    assert S.heuristic(900, 64, 148) == (S.LABEL_STREAMK, 160, 148, 0)
    assert S.heuristic(1024, 64, 132)[0] == S.LABEL_DP
    # iters <= min_iters stays data-parallel; whole waves stay data-parallel.
    assert S.heuristic(144, 8, 132)[0] == S.LABEL_DP
    assert S.heuristic(264, 64, 132)[0] == S.LABEL_DP
    # units dividing evenly over fewer tiles: Split-K label (4 tiles, 32 iters, 148 SMs
    # -> sk_units = min(148, 128 // 8 = 16) = 16 = 4 per tile).
    assert S.heuristic(4, 32, 148) == (S.LABEL_SPLITK, 4, 16, 4)


def _check_plan_invariants(p, M, N, K, sms):
    """Properties any correct plan has, checked by brute force over every iteration."""
    cover = {}
    for s in p.segments():
        assert 0 <= s.k_begin < s.k_end <= p.iters
        for k in range(s.k_begin, s.k_end):
            key = (s.tile, k)
            assert key not in cover, key
            cover[key] = s
    assert len(cover) == p.tiles * p.iters
    owners = {}
    for s in p.segments():
        if s.k_begin == 0:
            owners[s.tile] = s
    assert len(owners) == p.tiles
    for t, o in owners.items():
        contrib = [s for s in p.segments() if s.tile == t]
        if len(contrib) == 1:
            assert o.role in (S.FULL, S.SLAB) and o.k_end == p.iters
        elif o.role != S.SLAB:
            assert o.role == S.OWNER and o.n_peers == len(contrib) - 1
            peers = sorted((s for s in contrib if s is not o), key=lambda s: s.k_begin)
            assert [s.slot for s in peers] == list(range(o.peer_begin, o.peer_begin + o.n_peers))
            assert all(s.role == S.PRODUCER and s.peer_begin == o.peer_begin for s in peers)
    slots = [s.slot for s in p.segments() if s.role == S.PRODUCER]
    assert len(slots) == len(set(slots))
    assert all(0 <= x < p.n_slots for x in slots)


def test_streamk_bruteforce():
    # Every small flattened space: divmod ranges are contiguous, balanced within one
    # iteration, each unit has at most one producer (its first segment) and one owner (its
    # last), the owner of a split tile is its lowest contributor, and contributors are
    # consecutive units (n_contrib == u_last - u_first + 1, as in the Triton fixup).
    for tiles, iters, units in itertools.product(range(1, 13), range(1, 10), range(1, 30)):
        if units > tiles * iters:
            continue
        b = S.divmod_bounds(tiles * iters, units)
        sizes = [e - s for s, e in b]
        assert max(sizes) - min(sizes) <= 1 and sum(sizes) == tiles * iters
        assert all(b[i][1] == b[i + 1][0] for i in range(units - 1))
        segs = S._streamk_region(0, tiles, iters, units)
        for u, ss in enumerate(segs):
            roles = [s.role for s in ss]
            assert roles.count(S.PRODUCER) <= 1 and roles.count(S.OWNER) <= 1
            if S.PRODUCER in roles:
                assert roles[0] == S.PRODUCER
            if S.OWNER in roles:
                assert roles[-1] == S.OWNER
        for t in range(tiles):
            us = [u for u, (s, e) in enumerate(b) if s < (t + 1) * iters and e > t * iters]
            assert us == list(range(us[0], us[-1] + 1))
            owner = [s.unit for ss in segs for s in ss if s.tile == t and s.k_begin == 0]
            assert owner == [us[0]]


@pytest.mark.parametrize("mode", [S.DP, S.SPLITK, S.STREAMK, S.HYBRID])
def test_plan_invariants_small(mode):
    for M, N, K in [(128, 640, 256), (300, 200, 1000), (640, 640, 512), (128, 128, 64), (1, 1, 1)]:
        for sms in (1, 3, 4, 7, 16):
            splits = (1, 2, 3) if mode == S.SPLITK else (1,)
            for s in splits:
                if mode == S.SPLITK and s > S.problem_shape(M, N, K)[3]:
                    continue
                p = S.build_plan(M, N, K, sms, mode, splits=s)
                _check_plan_invariants(p, M, N, K, sms)
                if mode == S.SPLITK:
                    p2 = S.build_plan(M, N, K, sms, mode, splits=s, split_partials=1)
                    _check_plan_invariants(p2, M, N, K, sms)


@pytest.mark.parametrize("mode", [S.STREAMK, S.HYBRID])
def test_separate_fixup_slots(mode):
    # The separate fixup pass (first page, Case 3). The kernel there writes a unit's first
    # partial segment to slot 2u and a later one to 2u + 1. Its fixup_kernel finds tile t's
    # contributors u_first .. u_last from the range bounds and reads slot 2u if t is the
    # tile unit u's range starts in, else 2u + 1. That formula is written out here from the
    # bounds alone; the segment walk must produce exactly those slots, in k order, and
    # change nothing else.
    for M, N, K in [(128, 640, 256), (300, 200, 1000), (640, 640, 512), (128, 128, 64), (1, 1, 1),
                    (2048, 2432, 4096), (512, 512, 65536)]:
        for sms in (1, 3, 4, 7, 16, 148):
            for tile in (0, 2):
                if S.TILE_SHAPES[tile][2] > sms:
                    continue
                base = S.build_plan(M, N, K, sms, mode, tile=tile)
                sep = S.build_plan(M, N, K, sms, mode, tile=tile, split_partials=1)
                key = lambda q: [(x.unit, x.order, x.tile, x.k_begin, x.k_end, x.role) for x in q.segments()]
                assert key(sep) == key(base)
                if not sep.sk_tiles:  # the hybrid rule chose data-parallel: no partials
                    assert sep.n_slots == base.n_slots == 0 or sep.mode == S.DP
                    continue
                assert sep.n_slots == 2 * sep.sk_units
                iters = sep.iters
                bounds = S.divmod_bounds(sep.sk_tiles * iters, sep.sk_units)
                unit_of = lambda i: next(u for u, (b, e) in enumerate(bounds) if b <= i < e)
                want = {}
                for lt in range(sep.sk_tiles):
                    u_first, u_last = unit_of(lt * iters), unit_of((lt + 1) * iters - 1)
                    if u_first == u_last:
                        continue
                    want[sep.tiles - sep.sk_tiles + lt] = [
                        2 * u + (0 if bounds[u][0] // iters == lt else 1) for u in range(u_first, u_last + 1)]
                assert S.fixup_slots(sep) == want, (M, N, K, sms, tile)
                used = [x.slot for x in sep.segments() if x.role in (S.OWNER, S.PRODUCER)]
                assert len(used) == len(set(used)) and all(0 <= v < sep.n_slots for v in used)


def test_separate_fixup_rejected_where_meaningless():
    with pytest.raises(ValueError):
        S.build_plan(128, 640, 256, 4, S.DP, split_partials=1)
    with pytest.raises(ValueError):
        S.build_plan(128, 640, 256, 4, S.STREAMK, split_partials=2)


def test_splitk_clamped_and_dropped():
    # iters = 5, s = 4: chunk 2 -> splits [0,2) [2,4) [4,5); the empty fourth split is dropped.
    p = S.build_plan(128, 128, 320, 8, S.SPLITK, splits=4)
    assert p.splits == 3
    assert sorted((s.k_begin, s.k_end) for s in p.segments()) == [(0, 2), (2, 4), (4, 5)]
    with pytest.raises(ValueError):
        S.build_plan(128, 128, 320, 8, S.SPLITK, splits=6)


def test_splitk_producers_before_owner():
    # Many rounds of work items: a unit never waits on an item queued behind it.
    p = S.build_plan(1024, 1024, 1024, 5, S.SPLITK, splits=3)
    pos = {}
    for s in p.segments():
        pos[(s.tile, s.k_begin)] = (s.order * p.workers + s.unit)
    for s in p.segments():
        if s.role == S.OWNER:
            for q in p.segments():
                if q.tile == s.tile and q.role == S.PRODUCER:
                    assert pos[(q.tile, q.k_begin)] < pos[(s.tile, s.k_begin)]


def test_hybrid_waveq_on_148():
    # Wave-quantized shape: 16 x 19 = 304 tiles x 64 iterations on 148 SMs = 2 full waves + 8.
    p = S.build_plan(2048, 2432, 4096, 148, S.HYBRID)
    assert (p.tiles, p.iters) == (304, 64)
    assert p.mode == S.HYBRID and p.label == S.LABEL_STREAMK
    assert (p.sk_tiles, p.sk_units, p.workers) == (156, 148, 148)
    q, big = divmod(156 * 64, 148)
    assert (q, big) == (67, 68)
    assert max(c for _, c in S.tile_rows(p)) == 2
    dp_tiles = [s.tile for s in p.segments() if s.role == S.FULL and s.tile < 148]
    assert sorted(dp_tiles) == list(range(148))


def test_map_layout():
    p = S.build_plan(128, 640, 256, 4, S.STREAMK)
    m = S.plan_map(p)
    assert m[:S.HEADER_LEN] == [3, S.STREAMK, 5, 4, 4, 5, 4, 8, 0, -1, 0, 4, 128, 128, 1, 0, 0, 1]
    assert len(m) == S.HEADER_LEN + 8 * S.SEG_LEN + 5 * S.TILE_ROW_LEN
    # The toy's five tiles in one tile row, t at column t (the page's tile order).
    assert m[-5 * S.TILE_ROW_LEN:] == [0, 1, 0, 0, 0, 2, 0, 1, 1, 2, 0, 2, 2, 2, 0, 3, 3, 1, 0, 4]


@pytest.mark.parametrize("tile", [0, 1, 2, 3])
def test_tile_shapes(tile):
    # A pair tile is one unit of two SMs: 148 SMs give 74 units over 256-row tiles; the
    # wave-quantized shape keeps its 2 waves + a short tail (152 pair tiles on 74 units).
    tm, tn, cg = S.TILE_SHAPES[tile]
    p = S.build_plan(2048, 2432, 4096, 148, S.HYBRID, tile=tile)
    assert (p.tile_m, p.tile_n, p.cta_group) == (tm, tn, cg)
    assert p.tiles == S.cdiv(2048, tm) * S.cdiv(2432, tn)
    assert p.workers <= 148 // cg
    _check_plan_invariants(p, 2048, 2432, 4096, 148)
    if tile == 1:
        assert p.tiles == 152 and p.sk_units == 74 and p.sk_tiles == 152 - 74
    for mode in (S.DP, S.STREAMK, S.SPLITK):
        _check_plan_invariants(S.build_plan(300, 520, 1000, 7, mode, splits=2, tile=tile), 300, 520, 1000, 7)
    with pytest.raises(ValueError):
        S.build_plan(128, 128, 64, 1, S.DP, tile=1) if cg == 2 else S.build_plan(128, 128, 64, 1, S.DP, tile=9)


def test_rule_is_best_matches_printed_report():
    # The printed report (first page, Case 2): the rule's row equals the best of the four
    # schedules for 1536^2 on H100 and 3840^2 on B200, and loses to Split-K s = 4 at
    # 128 x 4096 and to Stream-K at 4096^2 on H100.
    want = {(1536, 1536, 132): True, (128, 4096, 132): False, (3840, 3840, 148): True, (4096, 4096, 132): False}
    for (m, n, sms), ok in want.items():
        c = S.schedule_choice(m, n, 4096, sms, 2, 2)
        assert c["rule_is_best"] is ok, (m, n, c)
    assert S.schedule_choice(128, 4096, 4096, 132, 2, 2)["best"] == 26.0


def _two_wave_list_schedule(item_costs, red_costs, sms):
    # Brute force: SMs take the next work item whenever they are free; the reduction
    # wave starts when every item of the first wave has finished.
    import heapq
    free = [0.0] * sms
    heapq.heapify(free)
    end = 0.0
    for c in item_costs:
        t = heapq.heappop(free) + c
        end = max(end, t)
        heapq.heappush(free, t)
    free = [end] * sms
    heapq.heapify(free)
    for c in red_costs:
        t = heapq.heappop(free) + c
        end = max(end, t)
        heapq.heappush(free, t)
    return end


@pytest.mark.parametrize("tiles,iters,sms,s", [(32, 64, 132, 2), (32, 64, 132, 4), (32, 64, 132, 8), (144, 64, 132, 4),
                                               (5, 4, 4, 2), (300, 16, 7, 4), (1, 64, 8, 16)])
@pytest.mark.parametrize("EPI,PART", [(2, 2), (2, 8), (0, 0), (3, 5)])
def test_split_k_separate_makespan_bruteforce(tiles, iters, sms, s, EPI, PART):
    # Splits divide iters here, so every item costs chunk + PART; each of the tiles'
    # reductions costs s * PART + EPI.
    chunk = iters // s
    items = [chunk + PART] * (tiles * s)
    reds = [s * PART + EPI] * tiles
    assert S.split_k_separate_makespan(tiles, iters, sms, s, EPI, PART) == _two_wave_list_schedule(items, reds, sms)


def test_rule_stops_best_scan():
    # Where the scan says the rule first stops being best after being best, check it by hand
    # from the page's rule and closed-form makespan bounds (EPI = PART = 2, 128 x 128 tiles,
    # 64 k-iterations, 132 SMs), not from the scan itself:
    #   m = 768: 6 * 32 = 192 tiles, tail 60, 2 * 60 < 132 -> the rule takes Stream-K;
    #   m = 896: 7 * 32 = 224 tiles, tail 92, 2 * 92 >= 132 -> the rule stays data-parallel,
    #            whose makespan is 2 waves * (64 + EPI) = 132;
    #   Stream-K at m = 896 puts 224 * 64 = 14336 iterations on 132 units, q = 108 (+1 for
    #   the first 80). A unit runs at most 109 iterations, holds at most one owner segment
    #   (EPI, plus PART per peer: a 109-iteration range meets at most 3 tiles of 64, so at
    #   most 2 peers) and at most one producer segment (PART), so it ends by
    #   109 + 2 + 2 * 2 + 2 = 117 < 132.
    tiles_896 = (896 // 128) * (4096 // 128)
    tail = tiles_896 - (tiles_896 // 132) * 132
    assert (tiles_896, tail) == (224, 92) and 2 * tail >= 132
    assert S.heuristic(tiles_896, 64, 132)[0] == S.LABEL_DP
    assert S.makespan(S.build_plan(896, 4096, 4096, 132, S.DP), 2, 2) == 2 * (64 + 2)
    assert S.makespan(S.build_plan(896, 4096, 4096, 132, S.STREAMK), 2, 2) <= 109 + 2 + 2 * 2 + 2
    assert S.heuristic(192, 64, 132)[0] == S.LABEL_STREAMK
    first, misses = S.rule_stops_best(range(128, 2049, 128), 4096, 4096, 132, 2, 2)
    # The scan's own contract: every miss is a shape where the rule's makespan exceeds the
    # best of the four, and `first` is the first miss that follows a hit.
    for m in misses:
        assert not S.schedule_choice(m, 4096, 4096, 132, 2, 2)["rule_is_best"]
    hits = [m for m in range(128, 2049, 128) if m not in misses]
    assert first == min(m for m in misses if m - 128 in hits)
    assert first == 896


def test_model_vs_gpu_report_fits_synthetic_timings(tmp_path, capsys):
    # The report's least-squares fit recovers a known unit: timings made from the model
    # itself at PART = 8 (10 us + 250 ns per k-iteration) fit exactly at PART = 8, and the
    # model then picks the fastest schedule on every shape.
    import json
    from oracle import model_vs_gpu as R
    ms = [128, 640, 1024, 2048]
    path = tmp_path / "exp.jsonl"
    with open(path, "w") as f:
        for m in ms:
            mr = R.model_rows(m, 8.0)
            for name in R.FOUR + ["rule"]:
                f.write(json.dumps({"experiment": "rule_vs_four", "M": m, "schedule": name,
                                    "us": 10.0 + 0.25 * mr[name]}) + "\n")
    R.main(str(path))
    out = capsys.readouterr().out
    assert f"PART=   8: model picks the measured best on {len(ms)}/{len(ms)} shapes" in out
    assert "fit us = 10.00 + 250.0 ns x makespan, rms relative error 0.0%" in out


def test_raster_default_is_the_page_tile_order():
    # First page, Case 3 listing: tile t covers rows (t // tiles_n) * BM and columns
    # (t % tiles_n) * BN. Raster 0 with no swizzle (0 or 1) is exactly that order.
    for M, N in [(640, 384), (2048, 2432), (128, 640), (1, 8), (4096, 4096)]:
        for sw in (0, 1):
            p = S.build_plan(M, N, 64, 4, S.DP, swizzle=sw)
            assert [S.tile_coords(p, t) for t in range(p.tiles)] == [divmod(t, p.tiles_n) for t in range(p.tiles)]


def test_raster_worked_examples():
    # 5 x 3 tiles (640 x 384), strips of 2. Along N: ids go down a 2-row strip, then along
    # N; the last strip (tile row 4) is one row deep. Along M: the transpose.
    p = S.build_plan(640, 384, 64, 4, S.DP, swizzle=2)
    assert [S.tile_coords(p, t) for t in range(15)] == [
        (0, 0), (1, 0), (0, 1), (1, 1), (0, 2), (1, 2), (2, 0), (3, 0), (2, 1), (3, 1), (2, 2), (3, 2),
        (4, 0), (4, 1), (4, 2)]
    p = S.build_plan(640, 384, 64, 4, S.DP, raster=1)
    assert [S.tile_coords(p, t) for t in range(15)] == [(t % 5, t // 5) for t in range(15)]
    p = S.build_plan(640, 384, 64, 4, S.DP, raster=1, swizzle=2)
    assert [S.tile_coords(p, t) for t in range(15)] == [
        (0, 0), (0, 1), (1, 0), (1, 1), (2, 0), (2, 1), (3, 0), (3, 1), (4, 0), (4, 1),
        (0, 2), (1, 2), (2, 2), (3, 2), (4, 2)]


def test_raster_is_a_bijection():
    for tm in (1, 2, 3, 5, 16, 17):
        for tn in (1, 2, 4, 7, 19):
            for raster in (0, 1):
                for sw in (0, 1, 2, 3, 4, 8, 16, 256):
                    p = S.build_plan(128 * tm, 128 * tn, 64, 4, S.DP, raster=raster, swizzle=sw)
                    got = [S.tile_coords(p, t) for t in range(p.tiles)]
                    assert sorted(got) == [(r, c) for r in range(tm) for c in range(tn)], (tm, tn, raster, sw)
