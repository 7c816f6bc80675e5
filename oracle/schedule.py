"""Schedule oracle: how the output tiles and their K loops are split over units.

TEST INFRASTRUCTURE (see the package docstring): plain, slow Python written from
the page "Split-K and Stream-K: The Last Wave of a GEMM" (kanthi.in), and, for the
Split-K factor heuristic, from the CUTLASS "Optimization Techniques" page. Every
function below names the passage it follows. Where a page leaves a step open, the
reading taken is stated at the function.

Terms (page, "Mental model" table): an output tile is BM x BN = 128 x 128; a
MAC-loop iteration is one BK = 64 step of a tile's K loop; a unit is one
persistent CTA (one per SM); the fixup combines a split tile's FP32 partials.

Map format produced by `plan_map` (int32 list), the contract the C library's
sk_plan must reproduce exactly:
  header (18): version, mode_resolved, tiles, iters, workers, sk_tiles, sk_units,
               n_segments, splits, label, label_splits, n_slots, tile_m, tile_n, cta_group,
               raster, swizzle, sk_groups
  n_segments rows (9): unit, order, tile, k_begin, k_end, role, slot, peer_begin, n_peers
  tiles rows (4): owner_unit, n_contrib, tile row, tile column
"""
from __future__ import annotations

from dataclasses import dataclass, field

TILE_M = 128
TILE_N = 128
BLK_K = 64

# decomposition modes (C-ABI enum values)
DP, SPLITK, STREAMK, HYBRID = 0, 1, 2, 3
# segment roles
FULL, OWNER, PRODUCER, SLAB = 0, 1, 2, 3
# heuristic labels
LABEL_NONE, LABEL_DP, LABEL_SPLITK, LABEL_STREAMK = -1, 0, 1, 2

# work-tile shapes: (tile_m, tile_n, CTAs per tile). A tile of the pair shapes is computed by
# two CTAs together, so a unit is a CTA pair and num_sms SMs give num_sms // 2 units.
TILE_SHAPES = {0: (128, 128, 1), 1: (256, 128, 2), 2: (256, 256, 2), 3: (128, 256, 1)}

MAP_VERSION = 3
HEADER_LEN = 18
SEG_LEN = 9
TILE_ROW_LEN = 4


def cdiv(a: int, b: int) -> int:
    return -(-a // b)


# ---------------------------------------------------------------------------
# Wave arithmetic (page, Case 1 "Count the waves before you tune anything")
# ---------------------------------------------------------------------------
def waves(m: int, n: int, sms: int, tile_m: int = TILE_M, tile_n: int = TILE_N):
    """Tiles, waves, CTAs in the final wave, and utilization tiles / (waves * SMs)."""
    tiles = cdiv(m, tile_m) * cdiv(n, tile_n)
    w = cdiv(tiles, sms)
    tail = tiles - (w - 1) * sms
    return tiles, w, tail, tiles / (w * sms)


def problem_shape(M: int, N: int, K: int, tile_m: int = TILE_M, tile_n: int = TILE_N):
    """Tile grid and K-loop length of a GEMM (page, Case 2 report: tiles and iters by ceiling)."""
    tiles_m, tiles_n = cdiv(M, tile_m), cdiv(N, tile_n)
    return tiles_m, tiles_n, tiles_m * tiles_n, cdiv(K, BLK_K)


# ---------------------------------------------------------------------------
# Unit ranges of the flattened (tile, k) space
# ---------------------------------------------------------------------------
def divmod_bounds(total: int, units: int):
    """Stream-K split (page, Case 2 stream_k_units; "Try this" calls it the CUTLASS split):
    q, big = divmod(total, units); the first `big` units take q + 1 iterations, the rest q."""
    q, big = divmod(total, units)
    out, it = [], 0
    for u in range(units):
        n = q + 1 if u < big else q
        out.append((it, it + n))
        it += n
    return out


def cdiv_bounds(total: int, units: int):
    """Variant of the page's Triton listing (Case 3): q = ceil(total / units), unit u owns
    [u*q, min((u+1)*q, total)). Documented variant only; the plans use divmod_bounds."""
    q = cdiv(total, units)
    return [(min(u * q, total), min((u + 1) * q, total)) for u in range(units)]


def floor_bounds(total: int, units: int):
    """Variant of the docc StreamK rewrite: block b owns [b*T/N, (b+1)*T/N) with floor division."""
    return [(b * total // units, (b + 1) * total // units) for b in range(units)]


# ---------------------------------------------------------------------------
# CUTLASS decision rule (page, Case 2 cutlass_heuristic; Case 4 knob table)
# ---------------------------------------------------------------------------
def heuristic(tiles: int, iters: int, sms: int, min_iters: int = 8):
    """Return (label, sk_tiles, sk_units, label_splits).

    Data-parallel when the tiles fill whole waves or the K loop is at most `min_iters`
    iterations, or when the tail wave is at least half full. Otherwise keep all full
    waves but the last data-parallel, give the remaining tiles to Stream-K over
    min(sms, iters * sk_tiles // min_iters) units, and call it Split-K when the units
    divide evenly over more than one per tile."""
    whole, tail = divmod(tiles, sms)          # full waves, and tiles left for a last one
    if tail == 0 or iters <= min_iters or 2 * tail >= sms:
        return LABEL_DP, 0, 0, 0
    dp_tiles = sms * max(whole - 1, 0)        # every full wave but the last stays DP
    sk_tiles = tiles - dp_tiles
    sk_units = min(sms, sk_tiles * iters // min_iters)
    per_tile, spare = divmod(sk_units, sk_tiles)
    if spare == 0 and per_tile > 1:
        return LABEL_SPLITK, sk_tiles, sk_units, per_tile
    return LABEL_STREAMK, sk_tiles, sk_units, 0


def calculate_split_k(m: int, n: int, k: int, num_sms: int) -> int:
    """Split-K factor heuristic (CUTLASS "Optimization Techniques" page, Split-K section,
    "Optimal Split-K Factor"). Count the whole 128 x 128 tiles of M x N (floor division, as
    printed); with at least two tiles per SM there is no split. Otherwise aim at four
    blocks per SM: the factor is the number of splits per tile that reaches 4 * num_sms
    blocks (rounded up), at most 32. K does not enter.

    Reading: a problem with fewer than 128 rows or columns has no whole tile, where the
    printed code would divide by zero; it counts as one tile here."""
    if m < 1 or n < 1 or num_sms < 1:
        raise ValueError("sizes and SM count must be positive")
    num_tiles = max(1, (m // 128) * (n // 128))
    if num_tiles >= 2 * num_sms:
        return 1
    target_blocks = 4 * num_sms
    return min(cdiv(target_blocks, num_tiles), 32)


def heuristic_text(label: int, sk_tiles: int, sk_units: int, label_splits: int) -> str:
    """The decision as the page's report prints it."""
    if label == LABEL_DP:
        return "DataParallel"
    name = f"SplitK(s={label_splits})" if label == LABEL_SPLITK else "StreamK"
    return f"{name} sk_tiles={sk_tiles} units={sk_units}"


# ---------------------------------------------------------------------------
# Work-unit plan
# ---------------------------------------------------------------------------
@dataclass
class Segment:
    unit: int
    order: int
    tile: int
    k_begin: int
    k_end: int
    role: int
    slot: int = -1
    peer_begin: int = -1
    n_peers: int = 0


@dataclass
class Plan:
    mode: int
    tiles: int
    iters: int
    tiles_n: int
    workers: int
    sk_tiles: int = 0
    sk_units: int = 0
    splits: int = 0
    label: int = LABEL_NONE
    label_splits: int = 0
    n_slots: int = 0
    units: list = field(default_factory=list)   # units[w] = list of Segment in execution order
    tile_m: int = TILE_M
    tile_n: int = TILE_N
    cta_group: int = 1
    tiles_m: int = 0
    raster: int = 0
    swizzle: int = 0
    sk_groups: int = 0   # groups the Stream-K region was split into (0: no Stream-K region)

    def segments(self):
        return [s for segs in self.units for s in segs]


def sk_group_count(n_tiles: int, iters: int, n_units: int, requested: int) -> int:
    """How many groups the Stream-K region is cut into (page, Case 4 knob table:
    `max_sk_groups_` caps the number of groups the Stream-K units form at 8, so that partials
    made at about the same time stay in L2). Reading taken: `requested` is that upper bound
    (0 or 1: one group). A group needs at least one tile and one unit, and no unit may be
    left without an iteration, so the count is the largest g <= min(requested, n_tiles,
    n_units) for which every group, tiles and units each divided big-first
    (group_bounds), has at least as many k-iterations as units."""
    g = min(max(1, requested), n_tiles, n_units)
    while g > 1:
        tb, ub = divmod_bounds(n_tiles, g), divmod_bounds(n_units, g)
        if all(u1 - u0 <= (t1 - t0) * iters for (t0, t1), (u0, u1) in zip(tb, ub)):
            return g
        g -= 1
    return 1


def group_bounds(n_tiles: int, iters: int, n_units: int, groups: int):
    """Flattened iteration range of every Stream-K unit when the region is cut into
    `groups` groups. Reading of the knob table's one sentence: the tiles of the region are
    divided into `groups` contiguous runs, and the units into as many consecutive groups,
    both big-first like the units of one region (the first n % g runs one larger); group j's
    units split only group j's run of tiles, by the divmod rule of stream_k_units (Case 2).
    With one group this is divmod_bounds(n_tiles * iters, n_units)."""
    out = []
    for (t0, t1), (u0, u1) in zip(divmod_bounds(n_tiles, groups), divmod_bounds(n_units, groups)):
        base = t0 * iters
        out += [(base + b, base + e) for b, e in divmod_bounds((t1 - t0) * iters, u1 - u0)]
    return out


def _streamk_region(tiles_base: int, n_tiles: int, iters: int, n_units: int, separate: bool = False,
                    groups: int = 1):
    """Per-unit segments of Stream-K over tiles [tiles_base, tiles_base + n_tiles).

    Follows the page's per-unit algorithm (Case 2 stream_k_units; Mental model): each unit
    walks its contiguous range of the flattened space one tile at a time. A segment that
    covers a whole tile is FULL. A segment that starts at the tile's k = 0 but stops short
    is the OWNER: it waits for the later units whose ranges start before the tile ends
    (its peers, in k order) and runs the fixup. Any other segment is a PRODUCER that stores
    an FP32 partial and raises a flag. Reading taken: each unit has one partial slot, its
    own index, so a tile's peers occupy consecutive slots owner+1 .. owner+n_peers.

    With `separate` (the page's Case 3 kernel: a separate fixup pass instead of waiting)
    every partial segment, the owner's too, stores to a fixed slot per (unit, first/last
    segment): slot 2u for the unit's first segment, 2u + 1 for a later one. Only a unit's
    first and last segments can be partial, and a producer is always its first.

    `groups` (at least 1, from sk_group_count): the unit ranges of group_bounds, so that no
    tile is shared between units of different groups."""
    bounds = group_bounds(n_tiles, iters, n_units, groups)
    starts = [b for b, _ in bounds]
    out = []
    for u in range(len(bounds)):
        b, e = bounds[u]
        segs = []
        if e > b:
            # The tiles the range [b, e) touches, and its piece of each.
            for local in range(b // iters, (e - 1) // iters + 1):
                t0 = local * iters
                kb, ke = max(b, t0) - t0, min(e, t0 + iters) - t0
                tile = tiles_base + local
                if (kb, ke) == (0, iters):
                    segs.append(Segment(u, 0, tile, kb, ke, FULL))
                elif kb == 0:
                    # Peers: the later units whose ranges begin inside the rest of the tile.
                    n_peers = sum(1 for v in range(u + 1, n_units) if starts[v] < t0 + iters)
                    slot = (2 * u + (0 if local == b // iters else 1)) if separate else -1
                    segs.append(Segment(u, 0, tile, kb, ke, OWNER, slot, u + 1, n_peers))
                else:
                    owner = next(v for v in range(u) if bounds[v][0] <= t0 < bounds[v][1])
                    segs.append(Segment(u, 0, tile, kb, ke, PRODUCER, 2 * u if separate else u, owner + 1, 0))
        out.append(segs)
    return out


def build_plan(M: int, N: int, K: int, num_sms: int, mode: int, splits: int = 1,
               units: int = 0, min_iters: int = 8, split_partials: int = 0, tile: int = 0,
               raster: int = 0, swizzle: int = 0, sk_groups: int = 0) -> Plan:
    """The integer work-unit map for one GEMM.

    `units` > 0 replaces num_sms as the number of persistent units (the toy case is
    "forced to 4 units"). Readings of the page where it leaves the step open:
      - DP (Mental model, Case 2 data_parallel): unit w runs tiles w, w + W, ... with
        W = min(units, tiles), each tile FULL.
      - Tile shape (`tile`, TILE_SHAPES): the pages' tile is 128 x 128 (tile 0). The
        CTA-pair shapes make one unit of two SMs, so `units` defaults to num_sms // 2; the
        schedule itself is the same over the coarser tile grid.
      - Split-K (Case 2 split_k; the split-K report's "final split is clamped"): split j
        of a tile covers k-iterations [j*chunk, min((j+1)*chunk, iters)), chunk =
        ceil(iters / s); empty trailing splits are dropped (s_eff = ceil(iters / chunk)).
        Split 0 owns the tile and reduces splits 1..s_eff-1 in k order. Work items are
        queued tile by tile with the owner last, item i -> tile i // s_eff, split
        s_eff-1 - i % s_eff, and unit w runs items w, w + W, ... (W = min(units, items)):
        every producer is queued before its owner, so no unit ever waits on work queued
        behind it. Slots: tile t's split j >= 1 uses slot t*(s_eff-1) + j-1.
        With split_partials (1 or 2) every split is a SLAB that writes its own [M,N] FP32
        slab j; 1 and 2 differ only in who sums the slabs, not in the plan.
      - Stream-K: units = min(units, tiles * iters) so that no unit is empty.
      - Hybrid (Case 2 hybrid; "gives the last 160 tiles ... to Stream-K"): the
        heuristic's Stream-K tiles are the last sk_tiles tile ids, split over sk_units
        units; the first tiles - sk_tiles run data-parallel over W units. Each unit runs
        its Stream-K range first, then its data-parallel tiles. A SplitK(s) label is
        planned with the same Stream-K partition (the page's hybrid simulates it so).
      - Stream-K and hybrid with split_partials = 1: the Stream-K tiles are merged by a
        separate fixup pass (Case 3), so every partial segment stores to its (unit,
        first/last) slot; see _streamk_region. A hybrid that resolves to DP has no partials.
      - sk_groups (Case 4 knob table, `max_sk_groups_`): the Stream-K region is cut into up
        to sk_groups groups of tiles and units (sk_group_count, group_bounds); 0 or 1 keeps
        one group, the plan of the page's simulator. Data-parallel and Split-K plans have
        no Stream-K region and ignore it.
    """
    if min(M, N, K) < 1 or num_sms < 1 or units < 0 or min_iters < 1:
        raise ValueError("bad problem")
    if mode not in (DP, SPLITK, STREAMK, HYBRID):
        raise ValueError("bad mode")
    if split_partials not in (0, 1, 2):
        raise ValueError("bad split_partials")
    if split_partials == 2 and mode != SPLITK:
        raise ValueError("the last-arriver sum needs Split-K slabs")
    if split_partials and mode == DP:
        raise ValueError("data-parallel tiles have no partials")
    if tile not in TILE_SHAPES:
        raise ValueError("bad tile shape")
    if raster not in (0, 1) or not 0 <= swizzle <= 256:
        raise ValueError("bad rasterization")
    if not 0 <= sk_groups <= 64:
        raise ValueError("bad sk_groups")
    tile_m, tile_n, cg = TILE_SHAPES[tile]
    tiles_m, tiles_n, tiles, iters = problem_shape(M, N, K, tile_m, tile_n)
    S = units if units > 0 else num_sms // cg
    if S < 1:
        raise ValueError("no units")
    p = _build(S, mode, splits, min_iters, split_partials, tiles, tiles_n, iters, sk_groups)
    p.tile_m, p.tile_n, p.cta_group = tile_m, tile_n, cg
    p.tiles_m, p.raster, p.swizzle = tiles_m, raster, swizzle
    return p


def tile_coords(p: Plan, t: int):
    """(tile row, tile column) of tile id t: the rasterization of the tile grid (the
    CUTLASS page, "Threadblock Rasterization": raster order along N or M, and a swizzle
    that keeps consecutive tiles in a band for L2 reuse). Reading taken: raster 0 walks the
    ids along N (row-major, the first page's tile order, tile t at row t // tiles_n); raster
    1 walks along M. A swizzle w >= 2 cuts the dimension across the walk into strips w
    tiles deep; ids fill one strip at a time, going across the strip's w tiles first and
    then along the walk. w = 0 or 1 is no swizzle."""
    across, along = (p.tiles_m, p.tiles_n) if p.raster == 0 else (p.tiles_n, p.tiles_m)
    w = max(1, p.swizzle)
    strip, i = divmod(t, w * along)
    h = min(w, across - strip * w)        # the last strip may be shallower
    a, b = strip * w + i % h, i // h      # position across and along the walk
    return (a, b) if p.raster == 0 else (b, a)


def _build(S, mode, splits, min_iters, split_partials, tiles, tiles_n, iters, sk_groups=0) -> Plan:
    if mode == HYBRID:
        label, sk_tiles, sk_units, lsp = heuristic(tiles, iters, S, min_iters)
        if label == LABEL_DP:
            p = _build(S, DP, 1, min_iters, 0, tiles, tiles_n, iters)
            p.label, p.label_splits = label, lsp
            return p
        dp_tiles = tiles - sk_tiles
        W = max(sk_units, min(S, dp_tiles))
        sep = bool(split_partials)
        p = Plan(HYBRID, tiles, iters, tiles_n, W, sk_tiles, sk_units, 0, label, lsp,
                 (2 if sep else 1) * sk_units)
        p.sk_groups = sk_group_count(sk_tiles, iters, sk_units, sk_groups)
        region = _streamk_region(dp_tiles, sk_tiles, iters, sk_units, sep, p.sk_groups)
        for w in range(W):
            segs = list(region[w]) if w < sk_units else []
            for t in range(w, dp_tiles, W):
                segs.append(Segment(w, 0, t, 0, iters, FULL))
            p.units.append(segs)
    elif mode == DP:
        W = min(S, tiles)
        p = Plan(DP, tiles, iters, tiles_n, W)
        for w in range(W):
            p.units.append([Segment(w, 0, t, 0, iters, FULL) for t in range(w, tiles, W)])
    elif mode == STREAMK:
        U = min(S, tiles * iters)
        sep = bool(split_partials)
        p = Plan(STREAMK, tiles, iters, tiles_n, U, tiles, U, 0, LABEL_NONE, 0, (2 if sep else 1) * U)
        p.sk_groups = sk_group_count(tiles, iters, U, sk_groups)
        p.units = _streamk_region(0, tiles, iters, U, sep, p.sk_groups)
    else:  # SPLITK
        if splits < 1 or splits > iters:
            raise ValueError("bad splits")
        chunk = cdiv(iters, splits)
        s_eff = cdiv(iters, chunk)
        items = tiles * s_eff
        W = min(S, items)
        n_slots = 0 if split_partials else tiles * (s_eff - 1)
        p = Plan(SPLITK, tiles, iters, tiles_n, W, 0, 0, s_eff, LABEL_NONE, 0, n_slots)
        for w in range(W):
            segs = []
            for i in range(w, items, W):
                t = i // s_eff
                j = s_eff - 1 - i % s_eff
                kb, ke = j * chunk, min((j + 1) * chunk, iters)
                if split_partials:
                    segs.append(Segment(w, 0, t, kb, ke, SLAB, j, -1, 0))
                elif s_eff == 1:
                    segs.append(Segment(w, 0, t, kb, ke, FULL))
                elif j == 0:
                    segs.append(Segment(w, 0, t, kb, ke, OWNER, -1, t * (s_eff - 1), s_eff - 1))
                else:
                    segs.append(Segment(w, 0, t, kb, ke, PRODUCER, t * (s_eff - 1) + j - 1,
                                        t * (s_eff - 1), 0))
            p.units.append(segs)
    for w, segs in enumerate(p.units):
        for i, s in enumerate(segs):
            s.unit, s.order = w, i
    return p


def fixup_slots(p: Plan):
    """For the separate fixup pass (Case 3 fixup_kernel): {tile: [slot, ...]} for every
    tile covered by more than one segment, the slots in ascending k order. The pass sums
    them left to right in FP32, the same order as the owner's turnstile."""
    by_tile = {}
    for s in p.segments():
        if s.role in (OWNER, PRODUCER):
            by_tile.setdefault(s.tile, []).append((s.k_begin, s.slot))
    return {t: [slot for _, slot in sorted(v)] for t, v in by_tile.items()}


def tile_rows(p: Plan):
    """Per tile: the unit that runs its k = 0 segment (the fixup owner) and the number of
    segments that cover it."""
    owner = [-1] * p.tiles
    n = [0] * p.tiles
    for s in p.segments():
        n[s.tile] += 1
        if s.k_begin == 0:
            owner[s.tile] = s.unit
    return list(zip(owner, n))


def plan_map(p: Plan):
    segs = p.segments()
    out = [MAP_VERSION, p.mode, p.tiles, p.iters, p.workers, p.sk_tiles, p.sk_units,
           len(segs), p.splits, p.label, p.label_splits, p.n_slots, p.tile_m, p.tile_n, p.cta_group,
           p.raster, p.swizzle, p.sk_groups]
    for s in segs:
        out += [s.unit, s.order, s.tile, s.k_begin, s.k_end, s.role, s.slot, s.peer_begin, s.n_peers]
    for t, (o, c) in enumerate(tile_rows(p)):
        out += [o, c, *tile_coords(p, t)]
    return out


# ---------------------------------------------------------------------------
# Cost model (page, Case 2: 1 per MAC-loop iteration, EPI per finished tile,
# PART per FP32 partial tile stored or loaded)
# ---------------------------------------------------------------------------
def makespan(p: Plan, EPI: float = 2.0, PART: float = 2.0) -> float:
    """Finish time of the slowest unit when every unit starts at 0 and runs its
    segments in order: a segment costs its iterations; a PRODUCER then pays PART to
    store its partial and signals; an OWNER waits for each peer's signal in k order,
    paying PART per partial loaded, then EPI; a FULL tile pays EPI."""
    signal = {}
    done = {}

    def unit_time(w):
        if w in done:
            return done[w]
        t = 0.0
        for s in p.units[w]:
            t += s.k_end - s.k_begin
            if s.role == PRODUCER:
                t += PART
                signal[s.slot] = t
            elif s.role == OWNER:
                for slot in range(s.peer_begin, s.peer_begin + s.n_peers):
                    if slot not in signal:
                        unit_time(_producer_unit(p, slot))
                    t = max(t, signal[slot]) + PART
                t += EPI
            elif s.role == SLAB:
                t += PART
            else:
                t += EPI
        done[w] = t
        return t

    return max(unit_time(w) for w in range(len(p.units))) if p.units else 0.0


def _producer_unit(p: Plan, slot: int) -> int:
    for s in p.segments():
        if s.role == PRODUCER and s.slot == slot:
            return s.unit
    raise KeyError(slot)


def split_k_makespan(tiles: int, iters: int, sms: int, s: int, EPI: float = 2.0, PART: float = 2.0):
    """The page's closed form for Split-K (Case 2 split_k): ceil(tiles*s / sms) waves of the
    worst unit (chunk iterations plus one partial store or load), then the owner's s-1
    further partial loads and the epilogue."""
    chunk = cdiv(iters, s)
    return cdiv(tiles * s, sms) * (chunk + PART) + (s - 1) * PART + EPI


def split_k_separate_makespan(tiles: int, iters: int, sms: int, s: int, EPI: float = 2.0, PART: float = 2.0):
    """Split-K whose reduction is its own wave of work (the page's "Try this": a Split-K
    variant with a separate reduction kernel). Reading taken: every split, split 0 too,
    stores its partial (chunk + PART per work item, ceil(tiles*s / sms) waves); then one
    reduction unit per tile loads its s partials and runs the epilogue (s*PART + EPI per
    unit, ceil(tiles / sms) waves). Nobody waits on anybody inside a wave."""
    chunk = cdiv(iters, s)
    return cdiv(tiles * s, sms) * (chunk + PART) + cdiv(tiles, sms) * (s * PART + EPI)


def schedule_choice(m: int, n: int, k: int, sms: int, EPI: float = 2.0, PART: float = 2.0):
    """The four schedules' makespans for one shape under (EPI, PART), the hybrid rule's
    label and makespan, and whether the rule's choice is (one of) the best of the four.
    Ties count as best."""
    rows = report_rows(m, n, k, sms, EPI, PART)[3]
    four = {name: t for name, t, _ in rows[:4]}
    rule_name, rule_t, _ = rows[4]
    best = min(four.values())
    return {"m": m, "four": four, "rule": rule_name, "rule_makespan": rule_t, "best": best,
            "rule_is_best": rule_t <= best + 1e-9}


def rule_stops_best(ms, n: int, k: int, sms: int, EPI: float = 2.0, PART: float = 2.0):
    """Scan m over `ms` (ascending): the first m at which the rule's choice is not the best
    of the four schedules after it was the best at the previous m (None if that never
    happens), and the list of every m where it is not the best."""
    prev, first, misses = None, None, []
    for m in ms:
        ok = schedule_choice(m, n, k, sms, EPI, PART)["rule_is_best"]
        if not ok:
            misses.append(m)
            if prev and first is None:
                first = m
        prev = ok
    return first, misses


def report_rows(m: int, n: int, k: int, sms: int, EPI: float = 2.0, PART: float = 2.0):
    """The five rows of the page's schedule report for one shape: (name, makespan, eff),
    plus the ideal makespan tiles * (iters + EPI) / sms."""
    _, _, tiles, iters = problem_shape(m, n, k)
    ideal = tiles * (iters + EPI) / sms
    rows = [("data-parallel", makespan(build_plan(m, n, k, sms, DP), EPI, PART))]
    for s in (2, 4):
        rows.append((f"split-K s={s}", split_k_makespan(tiles, iters, sms, s, EPI, PART)))
    rows.append(("stream-K (all tiles, 1 unit/SM)", makespan(build_plan(m, n, k, sms, STREAMK), EPI, PART)))
    hp = build_plan(m, n, k, sms, HYBRID)
    if hp.label == LABEL_DP:
        text = heuristic_text(LABEL_DP, 0, 0, 0)
    else:
        text = heuristic_text(hp.label, hp.sk_tiles, hp.sk_units, hp.label_splits)
    rows.append((f"CUTLASS heuristic -> {text}", makespan(hp, EPI, PART)))
    return tiles, iters, ideal, [(name, t, ideal / t) for name, t in rows]
