// sk_schedule.h - the work decomposition, shared by the host planner (sk_plan) and the
// persistent GEMM kernel. Both walk a unit's segments with SkWalk, so the map that
// sk_plan reports is, segment for segment, what each CTA executes.
//
// Sources: "Split-K and Stream-K: The Last Wave of a GEMM" (kanthi.in): Mental model
// (roles, k = 0 owner), Case 2 (data_parallel, split_k, stream_k_units,
// cutlass_heuristic, hybrid), Case 4 (decomposition modes). Readings where the page
// leaves a step open are stated at each branch.
#pragma once
#include <stdint.h>

#if defined(__CUDACC__)
#define SK_HD __host__ __device__ __forceinline__
#else
#define SK_HD inline
#endif

namespace sk {

// Division by a divisor fixed for the launch, as a multiply-high, an add and a shift (the
// "round-up" method of Hacker's Delight, chapter 10): with s = ceil(log2 d) and
// m = floor(2^32 (2^s - d) / d) + 1, n / d = (mulhi(n, m) + n) >> s for every 32-bit n. A
// hardware-less integer division costs tens of dependent instructions; the schedule walk
// divides by the same few numbers again and again, one thread at a time.
struct FastDiv {
    uint32_t d, m, s;
};
inline FastDiv make_fastdiv(uint32_t d) {
    FastDiv f{d > 0 ? d : 1u, 0u, 0u};
    while ((1ull << f.s) < f.d) ++f.s;
    f.m = static_cast<uint32_t>(((1ull << 32) * ((1ull << f.s) - f.d)) / f.d + 1);
    return f;
}

enum Mode : int32_t { kDP = 0, kSplitK = 1, kStreamK = 2, kHybrid = 3 };
enum Role : int32_t { kFull = 0, kOwner = 1, kProducer = 2, kSlab = 3 };
enum Label : int32_t { kLabelNone = -1, kLabelDP = 0, kLabelSplitK = 1, kLabelStreamK = 2 };

constexpr int32_t kTileM = 128;
constexpr int32_t kTileN = 128;
constexpr int32_t kBlkK = 64;

// Everything a unit needs to enumerate its segments; O(1) in size.
struct Sched {
    int32_t mode;          // resolved mode
    int32_t tiles, iters, tiles_n;
    int32_t workers;       // persistent units launched
    // Stream-K region: tiles [sk_base, sk_base + sk_tiles) over sk_units units. With one
    // group, unit u owns flattened iterations [u*q + min(u, big), (u+1)*q + min(u+1, big)).
    // With sk_groups > 1 (Case 4 knob table, max_sk_groups_) the region's tiles and units are
    // each cut big-first into sk_groups consecutive groups, and group j's units split only
    // group j's tiles by the same rule.
    int32_t sk_tiles, sk_units, sk_q, sk_big, sk_base, sk_groups;
    // Data-parallel region: tiles [0, dp_tiles), unit w runs w, w + workers, ...
    int32_t dp_tiles;
    // Split-K: effective split count, k-iterations per split, slab mode (1 reduction pass,
    // 2 in the one launch), and whether the splits of a tile share the sum (2, when every
    // work item has a unit of its own and so all splits of a tile run at once).
    int32_t splits, chunk, partials, coop;
    // Stream-K tiles merged by a separate fixup pass (every partial segment stores to slot
    // 2 * unit for the unit's first segment, 2 * unit + 1 for its last; nobody waits).
    int32_t sep;
    int32_t label, label_splits, n_slots;
    // Work-tile shape and CTAs per tile (a unit is one CTA or one CTA pair).
    int32_t tile_m, tile_n, cg;
    // Rasterization of the tile grid: tile ids walk along N (0) or M (1), in strips of
    // `swizzle` tiles across the walk (0 or 1: no strips).
    int32_t tiles_m, raster, swizzle;
    // Launch option, not part of the plan: overlap each launch with the kernel before it on
    // the stream (programmatic dependent launch; 2: and load A and B before it completes).
    int32_t overlap;
    // The walk's divisors: iters, sk_q + 1, sk_q (at least 1 wherever it is used), splits, and
    // for the tile order the strip size swizzle * (tiles along the walk) and the swizzle.
    FastDiv fd_iters, fd_q1, fd_q, fd_splits, fd_strip, fd_w;
};

// (tile_m, tile_n, CTAs per tile) of each sk_tile value; false for an unknown value.
SK_HD bool tile_shape(int32_t tile, int32_t* tm, int32_t* tn, int32_t* cg) {
    switch (tile) {
        case 0: *tm = 128; *tn = 128; *cg = 1; return true;
        case 1: *tm = 256; *tn = 128; *cg = 2; return true;
        case 2: *tm = 256; *tn = 256; *cg = 2; return true;
        case 3: *tm = 128; *tn = 256; *cg = 1; return true;
        default: return false;
    }
}

// Split-partials workspace: [0, 256) status | FP32 slabs [splits][M][N] from byte 256 |
// one arrival counter per tile and CTA of the tile from slab_counters_offset (256-aligned).
SK_HD int64_t slab_counters_offset(int32_t splits, int32_t M, int32_t N) {
    const int64_t end = 256 + 4ll * splits * M * N;
    return (end + 255) / 256 * 256;
}
SK_HD int64_t slab_workspace_bytes(int32_t splits, int32_t M, int32_t N, int32_t tiles, int32_t cg) {
    return slab_counters_offset(splits, M, N) + (4ll * tiles * cg + 255) / 256 * 256;
}

struct Seg {
    int32_t tile, k_begin, k_end, role, slot, peer_begin, n_peers;
};

SK_HD int32_t cdiv(int32_t a, int32_t b) { return (a + b - 1) / b; }
// n / f.d for 0 <= n < 2^31.
SK_HD int32_t fdiv(const FastDiv& f, int32_t n) {
    const uint32_t u = static_cast<uint32_t>(n);
#if defined(__CUDA_ARCH__)
    const uint32_t hi = __umulhi(u, f.m);
#else
    const uint32_t hi = static_cast<uint32_t>((static_cast<uint64_t>(u) * f.m) >> 32);
#endif
    return static_cast<int32_t>((static_cast<uint64_t>(hi) + u) >> f.s);
}
SK_HD int32_t imin(int32_t a, int32_t b) { return a < b ? a : b; }
SK_HD int32_t imax(int32_t a, int32_t b) { return a > b ? a : b; }

// (tile row, tile column) of tile id t ("Threadblock Rasterization" on the CUTLASS page:
// raster order along N or M, swizzled into bands for L2 reuse). With raster 0 and no
// swizzle, tile t sits at row t / tiles_n, column t % tiles_n (the first page's order). A
// swizzle w >= 2 cuts the dimension across the walk into strips w tiles deep; ids fill
// one strip at a time, across its (up to) w tiles first, then along the walk.
SK_HD void tile_coords(const Sched& s, int32_t t, int32_t* row, int32_t* col) {
    const int32_t across = s.raster == 0 ? s.tiles_m : s.tiles_n;
    const int32_t along = s.raster == 0 ? s.tiles_n : s.tiles_m;
    const int32_t w = s.swizzle > 1 ? s.swizzle : 1;
    const int32_t strip = fdiv(s.fd_strip, t);
    const int32_t i = t - strip * w * along;
    const int32_t h = imin(w, across - strip * w);
    const int32_t q = h == w ? fdiv(s.fd_w, i) : i / h;  // a full strip, or the last one
    const int32_t a = strip * w + (i - q * h);
    const int32_t b = q;
    *row = s.raster == 0 ? a : b;
    *col = s.raster == 0 ? b : a;
}

// n items cut into `parts` consecutive runs, the first n % parts runs one longer (the divmod
// split of Case 2 stream_k_units): the first item of run j, and the run holding item i.
// parts <= n, so every run is at least one long.
SK_HD int32_t run_begin(int32_t n, int32_t parts, int32_t j) { return j * (n / parts) + imin(j, n % parts); }
SK_HD int32_t run_of(int32_t n, int32_t parts, int32_t i) {
    const int32_t q = n / parts, big = n % parts, edge = big * (q + 1);
    return i < edge ? i / (q + 1) : big + (i - edge) / q;
}

// First flattened iteration of Stream-K unit u (divmod split, the first `big` units
// one iteration longer: Case 2 stream_k_units); u = sk_units gives the region's end.
// With groups: the unit's group, its place in the group, and the group's split.
SK_HD int32_t sk_unit_begin(const Sched& s, int32_t u) {
    if (s.sk_groups <= 1) return u * s.sk_q + imin(u, s.sk_big);
    if (u >= s.sk_units) return s.sk_tiles * s.iters;
    const int32_t g = s.sk_groups;
    const int32_t j = run_of(s.sk_units, g, u);
    const int32_t u0 = run_begin(s.sk_units, g, j), nu = run_begin(s.sk_units, g, j + 1) - u0;
    const int32_t t0 = run_begin(s.sk_tiles, g, j), nt = run_begin(s.sk_tiles, g, j + 1) - t0;
    return t0 * s.iters + run_begin(nt * s.iters, nu, u - u0);
}

// The unit whose range holds flattened iteration i.
SK_HD int32_t sk_unit_of(const Sched& s, int32_t i) {
    if (s.sk_groups <= 1) {
        const int32_t edge = s.sk_big * (s.sk_q + 1);
        return i < edge ? fdiv(s.fd_q1, i) : s.sk_big + fdiv(s.fd_q, i - edge);
    }
    const int32_t g = s.sk_groups;
    const int32_t j = run_of(s.sk_tiles, g, fdiv(s.fd_iters, i));
    const int32_t u0 = run_begin(s.sk_units, g, j), nu = run_begin(s.sk_units, g, j + 1) - u0;
    const int32_t t0 = run_begin(s.sk_tiles, g, j), nt = run_begin(s.sk_tiles, g, j + 1) - t0;
    return u0 + run_of(nt * s.iters, nu, i - t0 * s.iters);
}

// Groups actually used when up to `requested` are asked for: the largest g <= min(requested,
// tiles, units) for which every group has at least as many k-iterations as units, so that no
// unit is left empty (the knob table's "up to"); 0 or 1 gives one group.
SK_HD int32_t sk_group_count(int32_t tiles, int32_t iters, int32_t units, int32_t requested) {
    int32_t g = imin(imin(requested > 1 ? requested : 1, tiles), units);
    for (; g > 1; --g) {
        bool ok = true;
        for (int32_t j = 0; j < g && ok; ++j) {
            const int32_t nu = run_begin(units, g, j + 1) - run_begin(units, g, j);
            const int32_t nt = run_begin(tiles, g, j + 1) - run_begin(tiles, g, j);
            ok = static_cast<int64_t>(nu) <= static_cast<int64_t>(nt) * iters;
        }
        if (ok) break;
    }
    return g;
}

// Iterator over one unit's segments in run order: its Stream-K range first (if any),
// then its data-parallel tiles or Split-K work items.
struct Walk {
    int32_t unit;
    int32_t phase;   // 0: Stream-K range, 1: strided items, 2: done
    int32_t it, end; // Stream-K cursor / end, or the next item index

    SK_HD void init(const Sched& s, int32_t w) {
        unit = w;
        if ((s.mode == kStreamK || s.mode == kHybrid) && w < s.sk_units) {
            phase = 0;
            it = sk_unit_begin(s, w);
            end = sk_unit_begin(s, w + 1);
        } else {
            phase = 1;
            it = w;
            end = 0;
        }
    }

    SK_HD int32_t n_items(const Sched& s) const {
        return s.mode == kSplitK ? s.tiles * s.splits : s.dp_tiles;
    }

    SK_HD bool next(const Sched& s, Seg& g) {
        if (phase == 0) {
            if (it < end) {
                // One segment: the rest of the current tile inside this unit's range.
                const bool first = it == sk_unit_begin(s, unit);
                const int32_t local = fdiv(s.fd_iters, it);
                const int32_t tb = local * s.iters;
                const int32_t te = tb + s.iters;
                const int32_t se = imin(end, te);
                g.tile = s.sk_base + local;
                g.k_begin = it - tb;
                g.k_end = se - tb;
                g.slot = -1;
                g.peer_begin = -1;
                g.n_peers = 0;
                if (g.k_begin == 0 && g.k_end == s.iters) {
                    g.role = kFull;
                } else if (g.k_begin == 0) {
                    // k = 0 holder owns the fixup; its peers are the later units whose
                    // ranges start before the tile ends, i.e. up to the unit of te - 1.
                    g.role = kOwner;
                    g.peer_begin = unit + 1;
                    g.n_peers = sk_unit_of(s, te - 1) - unit;
                    if (s.sep) g.slot = 2 * unit + (first ? 0 : 1);
                } else {
                    // Partial handed to the owner; one slot per unit (its index). A producer
                    // is always its unit's first segment.
                    g.role = kProducer;
                    g.slot = s.sep ? 2 * unit : unit;
                    g.peer_begin = sk_unit_of(s, tb) + 1;
                }
                it = se;
                return true;
            }
            phase = 1;
            it = unit;
        }
        if (phase == 1) {
            if (it < n_items(s)) {
                g.slot = -1;
                g.peer_begin = -1;
                g.n_peers = 0;
                if (s.mode == kSplitK) {
                    // Work items queued tile by tile with the owner (split 0) last, so a
                    // unit never waits on an item queued behind it.
                    const int32_t t = fdiv(s.fd_splits, it);
                    const int32_t j = s.splits - 1 - (it - t * s.splits);
                    g.tile = t;
                    g.k_begin = j * s.chunk;
                    g.k_end = imin(g.k_begin + s.chunk, s.iters);
                    const int32_t base = t * (s.splits - 1);
                    if (s.partials) {
                        g.role = kSlab;
                        g.slot = j;
                    } else if (s.splits == 1) {
                        g.role = kFull;
                    } else if (j == 0) {
                        g.role = kOwner;
                        g.peer_begin = base;
                        g.n_peers = s.splits - 1;
                    } else {
                        g.role = kProducer;
                        g.slot = base + j - 1;
                        g.peer_begin = base;
                    }
                } else {
                    g.tile = it;
                    g.k_begin = 0;
                    g.k_end = s.iters;
                    g.role = kFull;
                }
                it += s.workers;
                return true;
            }
            phase = 2;
        }
        return false;
    }
};

}  // namespace sk
