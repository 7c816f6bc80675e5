// sk_kernels.cu - the persistent work-decomposed BF16 GEMM for sm_103a (the passes that sum
// partials in a second launch are in sk_passes.cu).
//
// One persistent unit per CTA, or per CTA pair for the pair tile shapes ("Split-K and
// Stream-K: The Last Wave of a GEMM", Mental model: one persistent CTA per SM, each
// walking its share of the flattened tile-by-k space). Each CTA walks its unit's segments
// (sk_schedule.h) with three roles:
//   warp 0      TMA producer: streams the A and B slabs of every k-iteration of every
//               segment into a shared-memory ring;
//   warp 1      MMA issuer: one thread issues tcgen05.mma (BF16 -> FP32) into one of two
//               TMEM accumulators, alternating per segment, so the epilogue of one segment
//               overlaps the MAC loop of the next. For a CTA pair only the leader (rank 0)
//               issues: tcgen05 cta_group::2 reads A rows and B columns from both CTAs'
//               shared memory and writes each CTA's rows into that CTA's TMEM;
//   warps 2..5  epilogue (and warps 6..9 with two epilogue groups): read the accumulator
//               from TMEM and act on the segment's role:
//               FULL -> write C; PRODUCER -> store the FP32 partial to its workspace slot
//               and raise a flag (or add it atomically and bump a counter); OWNER -> wait
//               for its peers in k order, add their partials, write C (Mental model;
//               Case 4 reduction modes). With the separate fixup pass (Case 3) OWNER and
//               PRODUCER both store to their (unit, first/last) slot and nobody waits.
//               SLAB -> write the split's FP32 [M,N] slab; with the in-launch sum, count
//               the arrival and sum a share of the tile (or, arriving last, all of it).
// Every wait is bounded by a deadline; on expiry the CTA records SK_ETIMEOUT in the
// workspace status word, unwinds its pipeline and returns.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "sk_kernels.h"
#include "sk_ptx.cuh"

namespace sk {

namespace {

constexpr int32_t kErrTimeout = -4;  // SK_ETIMEOUT
constexpr int32_t kErrBounds = -7;   // SK_EBOUNDS
constexpr uint64_t kDrainNs = 20ull * 1000 * 1000;

template <class S>
struct Smem {
    uint32_t base;  // shared address of the 1024-aligned ring
    __device__ uint32_t a(int s) const { return base + s * S::kABytes; }
    __device__ uint32_t b(int s) const { return base + S::kStages * S::kABytes + s * S::kBBytes; }
    __device__ uint32_t full(int s) const { return base + S::kSmemBarOff + 8 * s; }
    __device__ uint32_t empty(int s) const { return base + S::kSmemBarOff + 8 * (S::kStages + s); }
    __device__ uint32_t tfull(int b) const { return base + S::kSmemBarOff + 8 * (2 * S::kStages + b); }
    __device__ uint32_t tempty(int b) const { return base + S::kSmemBarOff + 8 * (2 * S::kStages + 2 + b); }
    __device__ uint32_t done() const { return base + S::kSmemBarOff + 8 * (2 * S::kStages + 4); }
    __device__ uint32_t tready() const { return base + S::kSmemBarOff + 8 * (2 * S::kStages + 5); }
    // Epilogue warp w's two barriers for partials fetched into the ring by bulk copies.
    __device__ uint32_t pload(int w, int b) const { return base + S::kSmemBarOff + kBarPload + 8 * (2 * w + b); }
};

// Ring bytes an epilogue warp may use once the unit's MAC loop is over (the ring split four ways).
constexpr uint32_t kWarpRingBytes = kRingBytes / 4;
// One pass of an epilogue warp's block of a partial (32 rows x kPassCols FP32): the unit of the
// bulk copies that bring a deterministic owner's peer partials into the ring.
constexpr uint32_t kPartBytes = 32u * kPassCols * 4u;
static_assert(2 * kPartBytes + 4 * 4096 <= kWarpRingBytes && 12 * 4096 <= kWarpRingBytes, "ring quarter");
// Shared-memory word that hands the first partial copies of the unit's last (owner) segment
// from the producer warp to the epilogue: 0 open; kPrefetchClosed once the epilogue has given
// up on the segment (the producer must not start copies any more); kPrefetchIssued + k once
// the producer started k copies per epilogue warp.
constexpr int kPrefetchClosed = 1;
constexpr int kPrefetchIssued = 2;



__device__ __forceinline__ void record_timeout(const KArgs& a, volatile int* abort_flag) {
    *abort_flag = 1;
    atomicCAS(a.status, 0, kErrTimeout);
}

// Where a CTA sits in its work tile: `rank` in its MMA pair (0 = the pair's leader, which
// issues the MMAs; its rows are rank * 128 .. of the tile, and its block of every partial
// slot and its flag are number `rank`). One-CTA tiles: zero.
struct CtaPos {
    uint32_t rank;
};

// A Stream-K producer segment covers [k_begin, iters) of its tile: it runs its k-loop from
// the last k-iteration down, so that all units start on the same k-slab of A and B (shared
// through L2) instead of each on its own (an HBM burst of every unit's data at once when
// the caches are cold). The order of the MMAs inside one segment's accumulator is free;
// the k order of the fold across segments is unchanged.
__device__ __forceinline__ bool reversed_segment(const Sched& s, const Seg& g) {
    return g.role == kProducer && g.k_end == s.iters;
}
__device__ __forceinline__ int32_t seg_k(const Seg& g, bool rev, int32_t i) {
    return rev ? g.k_end - 1 - i : g.k_begin + i;
}

// --------------------------------------------------------------------------- warp 0
// The unit's last segment g is a deterministic owner's (its peers' partials are summed in k
// order by the epilogue): acquire the peers' flags; once every load of the unit (`issued` of
// them) has been consumed by the MAC loop, the ring is free, so start the first one or two
// partial copies of each epilogue warp into its ring quarter, while the epilogue is still
// storing the segment before. Returns false when a wait gave up.
// The MMA issuer commits each stage's empty barrier after that stage's MMAs, and a commit
// arrives only once every MMA issued before it has completed, so the last load's stage
// turning empty means every stage has been read: one wait, not one per stage (each wait
// costs about 0.13 us even on a phase long complete). Issuing each copy as soon as the
// stages under its own buffer were free for good was measured too: no faster.
template <int kCG, int kBN>
__device__ bool prefetch_partials(const KArgs& a, const Smem<Shape<kCG, kBN>>& sm, const Seg& g, const CtaPos& pos,
                                  uint32_t issued, uint64_t deadline, volatile int* abort_flag, int* prefetch) {
    using S = Shape<kCG, kBN>;
    // Indices outside the workspace: leave the segment to the epilogue, which reports them.
    if (g.tile < 0 || g.tile >= a.sch.tiles || g.peer_begin < 0 || g.n_peers < 1 ||
        g.peer_begin + g.n_peers > a.sch.n_slots)
        return true;
    for (int32_t pi = 0; pi < g.n_peers; ++pi) {
        const int32_t* f = a.flags + (g.peer_begin + pi) * a.sch.cg + static_cast<int>(pos.rank);
        for (uint32_t n = 0; ld_acquire_gpu(f) < 1; ++n) {
            if ((n & 15u) == 15u && (*abort_flag || globaltimer() > deadline)) return false;
            __nanosleep(32);
        }
    }
    // Load n went to stage n % kStages; its consumption completes that stage's empty phase
    // n / kStages.
    if (issued > 0) {
        const uint32_t n = issued - 1;
        if (!mbar_wait(sm.empty(n % S::kStages), (n / S::kStages) & 1u, abort_flag, deadline)) return false;
    }
    const int k = S::kPasses * g.n_peers > 1 ? 2 : 1;
    if (atomicCAS(prefetch, 0, kPrefetchIssued + k) != 0) return true;  // the epilogue has given up
    fence_proxy_async_global();  // the flag acquires before the copies' reads
    for (int ew = 0; ew < 4; ++ew)
        for (int j = 0; j < k; ++j) fetch_partial(a, sm, g, static_cast<int>(pos.rank), ew, j);
    return true;
}

// An overlapped launch, before its wait for the previous kernel: prefetch into L2 the A and B
// boxes of the unit's first kStages loads (the ones run_producer issues first), so that they
// come from L2 instead of HBM once the wait is over. A prefetch has no effect on what later
// loads read: if the previous kernel writes these bytes, L2 holds its writes.
template <bool kNT, int kCG, int kBN>
__device__ void prefetch_first_loads(const KArgs& a, const CUtensorMap* tmA, const CUtensorMap* tmB, int unit,
                                     const CtaPos& pos) {
    using S = Shape<kCG, kBN>;
    Walk w;
    w.init(a.sch, unit);
    Seg g;
    int n = 0;
    while (n < S::kStages && w.next(a.sch, g)) {
        int32_t trow, tcolumn;
        tile_coords(a.sch, g.tile, &trow, &tcolumn);
        const int32_t m0 = trow * (kCtaRows * kCG) + static_cast<int32_t>(pos.rank) * kCtaRows;
        const int32_t nb = tcolumn * a.sch.tile_n + static_cast<int32_t>(pos.rank) * S::kBNc;
        const bool rev = reversed_segment(a.sch, g);
        for (int32_t i = 0; i < g.k_end - g.k_begin && n < S::kStages; ++i, ++n) {
            const int32_t k0 = seg_k(g, rev, i) * kBlkK;
            tma_prefetch_2d(tmA, k0, m0);
            if (kNT) {
                tma_prefetch_2d(tmB, k0, nb);
            } else {
#pragma unroll
                for (int j = 0; j < S::kBNc / 64; ++j) tma_prefetch_2d(tmB, nb + 64 * j, k0);
            }
        }
    }
}

template <bool kNT, int kCG, int kBN>
__device__ void run_producer(const KArgs& a, const CUtensorMap* tmA, const CUtensorMap* tmB,
                             const Smem<Shape<kCG, kBN>>& sm, Walk w, Seg g, bool have, const CtaPos& pos,
                             uint64_t deadline, volatile int* abort_flag, int* prefetch, bool early) {
    using S = Shape<kCG, kBN>;
    const uint32_t rank = pos.rank;
    Seg last;
    int nseg = 0;
    int stage = 0;
    uint32_t phase = 0;
    uint32_t issued = 0;
    bool ok = true;
    for (; ok && have; have = w.next(a.sch, g)) {
        if (early && nseg == 2) {
            // Operand loads ahead of the previous kernel (overlap = 2): the first two segments
            // fill the two fresh accumulators. The third waits on the epilogue, which waits for
            // that kernel, so from here on this warp waits for it too and its wait limits count
            // from then.
            grid_dep_wait();
            early = false;
            deadline = globaltimer() + a.timeout_ns;
        }
        last = g;
        ++nseg;
        // This CTA's rows of the tile and its half of the tile's columns of B.
        int32_t trow, tcolumn;
        tile_coords(a.sch, g.tile, &trow, &tcolumn);
        const int32_t m0 = trow * (kCtaRows * kCG) + static_cast<int32_t>(rank) * kCtaRows;
        const int32_t nb = tcolumn * a.sch.tile_n + static_cast<int32_t>(rank) * S::kBNc;
        const bool rev = reversed_segment(a.sch, g);
        for (int32_t i = 0; i < g.k_end - g.k_begin; ++i) {
            if (!mbar_wait(sm.empty(stage), phase ^ 1u, abort_flag, deadline)) {
                ok = false;
                break;
            }
            const int32_t k0 = seg_k(g, rev, i) * kBlkK;
            if (kCG == 1) {
                mbar_arrive_expect_tx(sm.full(stage), S::kTxBytes);
                tma_load_2d(sm.a(stage), tmA, sm.full(stage), k0, m0);
                if (kNT) {
                    tma_load_2d(sm.b(stage), tmB, sm.full(stage), k0, nb);
                } else {
#pragma unroll
                    for (int j = 0; j < S::kBNc / 64; ++j)
                        tma_load_2d(sm.b(stage) + j * 8192, tmB, sm.full(stage), nb + 64 * j, k0);
                }
            } else {
                // Both CTAs' loads complete on the leader's barrier, which the leader arms
                // for the bytes of both.
                const uint32_t fb = mapa_shared(sm.full(stage), 0u);
                if (rank == 0) mbar_arrive_expect_tx(sm.full(stage), S::kTxBytes);
                tma_load_2d_pair(sm.a(stage), tmA, fb, k0, m0);
                if (kNT) {
                    tma_load_2d_pair(sm.b(stage), tmB, fb, k0, nb);
                } else {
#pragma unroll
                    for (int j = 0; j < S::kBNc / 64; ++j)
                        tma_load_2d_pair(sm.b(stage) + j * 8192, tmB, fb, nb + 64 * j, k0);
                }
            }
            ++issued;
            if (++stage == S::kStages) {
                stage = 0;
                phase ^= 1u;
            }
        }
    }
    // The workspace (flags, partial slots, status word) is touched only after the previous
    // kernel has completed; the owner's partial fetch then waits within a limit counted
    // from there.
    if (early) {
        grid_dep_wait();
        deadline = globaltimer() + a.timeout_ns;
    }
    if (ok && kEpiGroups == 1 && nseg > 0 && last.role == kOwner && !a.sch.sep && !a.atomic)
        ok = prefetch_partials<kCG, kBN>(a, sm, last, pos, issued, deadline, abort_flag, prefetch);
    if (!ok) record_timeout(a, abort_flag);
    // Let the last loads land before the CTA can exit (bounded). A pair's loads all complete
    // on the leader's barriers, so the leader drains for both.
    if (rank == 0) {
        const uint64_t drain = globaltimer() + kDrainNs;
        const uint32_t outstanding = issued < static_cast<uint32_t>(S::kStages) ? issued : S::kStages;
        for (uint32_t i = 0; i < outstanding; ++i) {
            const uint32_t pos = issued - 1 - i;
            if (!mbar_wait_until(sm.full(pos % S::kStages), (pos / S::kStages) & 1u, drain)) break;
        }
    }
}

// --------------------------------------------------------------------------- warp 1
// The leader of each pair issues its pair's MMAs. Its commits reach both CTAs of the pair
// (cluster ranks 0 and 1) through a cluster-multicast mbarrier arrive.
template <bool kNT, int kCG, int kBN>
__device__ void run_mma(const KArgs& a, const Smem<Shape<kCG, kBN>>& sm, uint32_t tmem_base, Walk w, Seg g,
                        bool have, uint64_t deadline, volatile int* abort_flag, bool early) {
    using S = Shape<kCG, kBN>;
    constexpr uint16_t pair_mask = 0x3u;
    constexpr uint32_t kIdesc = idesc_bf16_f32(kCtaRows * kCG, kBN, kNT ? 0u : 1u);
    // K advance per 16-deep MMA inside one 64-deep stage: K-major operands move 32 bytes
    // along the swizzled row; the MN-major B of NN moves 16 rows of 128 bytes.
    constexpr uint32_t kAStep = (16 * 2) >> 4;
    constexpr uint32_t kBStep = kNT ? ((16 * 2) >> 4) : ((16 * 128) >> 4);
    int stage = 0;
    uint32_t phase = 0;
    int buf = 0;
    uint32_t uses0 = 0u, uses1 = 0u;  // phase parities of the two accumulators
    bool ok = true;
    uint64_t* tr = a.trace ? a.trace + static_cast<int64_t>(blockIdx.x) * kTraceWords : nullptr;
    int seg = 0;
    // A pair's MMA writes both CTAs' TMEM: wait until the peer has allocated its part.
    if (kCG == 2 && !mbar_wait<true>(sm.tready(), 0u, abort_flag, deadline)) ok = false;
    for (; ok && have; have = w.next(a.sch, g)) {
        if (early && seg == 2) {
            // As in the producer (overlap = 2): the third segment reuses the first accumulator,
            // which the epilogue hands back only after its own wait for the previous kernel.
            grid_dep_wait();
            early = false;
            deadline = globaltimer() + a.timeout_ns;
        }
        if (!mbar_wait<kCG == 2>(sm.tempty(buf), (buf ? uses1 : uses0) ^ 1u, abort_flag, deadline)) {
            ok = false;
            break;
        }
        tc_fence_after();
        const uint32_t d = tmem_base + static_cast<uint32_t>(buf * kBN);
        const int32_t len = g.k_end - g.k_begin;
        // Several stages per turn: one wait covers all of them (their barrier round trips
        // overlap), then four MMAs and a commit per stage. Three for an 8-stage ring, two for
        // a 6-stage one, one for the 128 x 256 tile's four stages of 48 KiB; a deeper turn on a
        // shallower ring leaves too few stages loading while the issuer waits. A segment's
        // last stages form a shorter turn.
        constexpr int kTurn = S::kStages >= 8 ? 3 : (S::kStages >= 6 ? 2 : 1);
        for (int32_t i = 0; i < len;) {
            const int nt = len - i < kTurn ? len - i : kTurn;
            uint32_t tb[3], tp[3];
            {
                int st = stage;
                uint32_t ph = phase;
#pragma unroll
                for (int h = 0; h < 3; ++h) {
                    tb[h] = sm.full(st);
                    tp[h] = ph;
                    if (++st == S::kStages) {
                        st = 0;
                        ph ^= 1u;
                    }
                }
            }
            const bool got = nt == 1 ? mbar_wait(tb[0], tp[0], abort_flag, deadline)
                                     : mbar_wait_n(nt, tb, tp, abort_flag, deadline);
            if (!got) {
                ok = false;
                break;
            }
            tc_fence_after();
            if (tr && i == 0 && seg < kTraceSegs) tr[4 + 4 * seg] = globaltimer();
#pragma unroll
            for (int h = 0; h < 3; ++h) {
                if (h >= nt) break;
                // A: K-major, 8-row groups 1024 bytes apart. B: K-major likewise (NT), or
                // MN-major (NN) in 64-column boxes 8 KiB apart.
                const uint64_t adesc = smem_desc_sw128(sm.a(stage), 16, 1024);
                const uint64_t bdesc =
                    kNT ? smem_desc_sw128(sm.b(stage), 16, 1024) : smem_desc_sw128(sm.b(stage), 8192, 1024);
#pragma unroll
                for (int kk = 0; kk < kBlkK / 16; ++kk) {
                    const uint32_t acc = (i + h > 0 || kk > 0) ? 1u : 0u;
                    if (kCG == 1)
                        umma_bf16(d, adesc + kk * kAStep, bdesc + kk * kBStep, kIdesc, acc);
                    else
                        umma_bf16_pair(d, adesc + kk * kAStep, bdesc + kk * kBStep, kIdesc, acc);
                }
                if (kCG == 1)
                    umma_commit(sm.empty(stage));
                else
                    umma_commit_pair(sm.empty(stage), pair_mask);
                if (++stage == S::kStages) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
            i += nt;
        }
        if (!ok) break;
        if (kCG == 1)
            umma_commit(sm.tfull(buf));
        else
            umma_commit_pair(sm.tfull(buf), pair_mask);
        if (tr && seg < kTraceSegs) tr[4 + 4 * seg + 1] = globaltimer();
        ++seg;
        if (buf)
            uses1 ^= 1u;
        else
            uses0 ^= 1u;
        buf ^= 1;
    }
    if (!ok) {
        if (early) grid_dep_wait();  // the status word is written after the previous kernel
        record_timeout(a, abort_flag);
    }
    // Every MMA issued so far has finished reading shared memory and writing TMEM (of
    // both CTAs of a pair) before this thread moves on to the exit barrier.
    if (kCG == 1)
        umma_commit(sm.done());
    else
        umma_commit_pair(sm.done(), static_cast<uint16_t>(0x1u));
    mbar_wait_until(sm.done(), 0u, globaltimer() + kDrainNs);
}

// --------------------------------------------------------------------------- warps 2..5
// Wait until *f >= target: lane 0 polls, then every lane performs its own acquire load.
__device__ __forceinline__ bool wait_flag(const int32_t* f, int32_t target, uint64_t deadline,
                                          const volatile int* abort_flag) {
    bool ok = true;
    if ((threadIdx.x & 31) == 0) {
        for (uint32_t n = 0;; ++n) {
            if (ld_acquire_gpu(f) >= target) break;
            if ((n & 15u) == 15u && (*abort_flag || globaltimer() > deadline)) {
                ok = false;
                break;
            }
            __nanosleep(32);
        }
    }
    // The warp's decision is lane 0's; each lane then takes its own acquire of the flag
    // (a bounded re-read that cannot change the decision).
    ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
    if (ok) {
        for (uint32_t n = 0; n < (1u << 20) && ld_acquire_gpu(f) < target; ++n) {
        }
    }
    return ok;
}

// Partial-slot layout: a CTA's share of a slot (128 rows x kBN columns FP32) is split into
// one contiguous block per TMEM lane quadrant (its 32 rows x kBN columns, block index quad);
// inside a block, element (lane, column 32c + 4q + e) sits at float4 index
// (c * 8 + q) * 32 + lane, so each warp access covers 512 contiguous bytes.
__device__ __forceinline__ int slot_f4(int c, int q, int lane) { return ((c * 8 + q) * 32 + lane) * 4; }

// Lane 0 of epilogue warp `ew`: fetch item j of a deterministic owner's peer partials (pass
// j / n_peers of peer j % n_peers, this warp's block) into the warp's ring buffer j % 2 with one
// bulk copy, completing on that buffer's barrier. Warp ew + 2 reads TMEM lane quadrant
// (ew + 2) % 4, whose rows are block (ew + 2) % 4 of the slot.
template <class S>
__device__ __forceinline__ void fetch_partial(const KArgs& a, const Smem<S>& sm, const Seg& g, int cta, int ew, int j) {
    constexpr int kChunks = kPassCols / 32;
    const int p = j / g.n_peers, pi = j % g.n_peers;
    const int quad = (ew + 2) & 3;
    const float* src = a.slots + static_cast<int64_t>((g.peer_begin + pi) * a.sch.cg + cta) * S::kCtaSlotFloats +
                       static_cast<int64_t>(quad) * S::kWarpSlotFloats + slot_f4(kChunks * p, 0, 0);
    const uint32_t bar = sm.pload(ew, j & 1);
    mbar_arrive_expect_tx(bar, kPartBytes);
    bulk_load_g2s(sm.base + static_cast<uint32_t>(ew) * kWarpRingBytes + static_cast<uint32_t>(j & 1) * kPartBytes,
                  src, kPartBytes, bar);
}

// Store kCols columns of this warp's 32 rows (one row per lane, in registers) through the
// warp's two 4 KiB staging boxes with TMA tensor stores: BF16 C in boxes of 64 columns, FP32
// C or slab in boxes of 32 columns, each box 32 rows x 128 bytes in the 128-byte swizzled
// layout (16-byte chunk j of row r at chunk j ^ (r % 8)), so the shared stores are
// conflict-free and the TMA clips the box at M and N. `slab` < 0 stores to C.
// Staging buffer of this warp's nstore-th box: the nbuf 4 KiB buffers at `staging` in
// turn (nbuf is 1, 2, 4 or 12). Before a buffer is reused, wait until the TMA has read the
// copy issued nbuf boxes ago.
__device__ __forceinline__ uint32_t staging_buffer(uint32_t staging, uint32_t nbuf, uint32_t nstore) {
    if (nstore >= nbuf) {
        if ((threadIdx.x & 31) == 0) {
            switch (nbuf) {
                case 1: bulk_wait_group_read<0>(); break;
                case 2: bulk_wait_group_read<1>(); break;
                case 4: bulk_wait_group_read<3>(); break;
                default: bulk_wait_group_read<11>(); break;
            }
        }
        __syncwarp();
    }
    return staging + (nstore % nbuf) * 4096u;
}

// One 32-row x 128-byte box of this warp's rows (8 chunks of 16 bytes per row, given as
// 32-bit words w[j][0..3]) through staging buffer nstore % nbuf, stored by the TMA at
// (x, y0) (or (x, y0, slab)).
template <class F>
__device__ __forceinline__ void store_box(const CUtensorMap* tmC, uint32_t staging, uint32_t nbuf, uint32_t& nstore,
                                          int32_t x, int32_t y0, int32_t slab, F&& words) {
    const int lane = threadIdx.x & 31;
    const uint32_t buf = staging_buffer(staging, nbuf, nstore);
    const uint32_t row = buf + static_cast<uint32_t>(lane) * 128u;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        uint32_t w0, w1, w2, w3;
        words(j, w0, w1, w2, w3);
        st_shared_v4(row + static_cast<uint32_t>((j ^ (lane & 7)) * 16), w0, w1, w2, w3);
    }
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) {
        if (slab < 0)
            tma_store_2d(tmC, buf, x, y0);
        else
            tma_store_3d(tmC, buf, x, y0, slab);
        bulk_commit_group();
    }
    ++nstore;
}

// Store kCols columns of this warp's 32 rows (one row per lane, in registers) with TMA
// tensor stores through the warp's 4 KiB staging boxes: BF16 C in boxes of 64 columns,
// FP32 C or slab in boxes of 32 columns, each box 32 rows x 128 bytes in the 128-byte
// swizzled layout (16-byte chunk j of row r at chunk j ^ (r % 8)), so the shared stores are
// conflict-free and the TMA clips the box at M and N. `slab` < 0 stores to C.
template <int kCols>
__device__ __forceinline__ void store_slice(const KArgs& a, const CUtensorMap* tmC, uint32_t staging, uint32_t nbuf,
                                            uint32_t& nstore, const float (&v)[kCols], int32_t x0, int32_t y0,
                                            int32_t slab) {
    if (y0 >= a.M) return;  // the warp's 32 rows lie below C
    if (x0 < 0 || y0 < 0) {  // never reached by a valid plan: record it and skip the stores
        atomicCAS(a.status, 0, kErrBounds);
        return;
    }
    if (a.c_bf16 && slab < 0) {
#pragma unroll
        for (int b = 0; b < kCols / 64; ++b) {
            const int32_t x = x0 + b * 64;
            if (x >= a.N) break;
            store_box(tmC, staging, nbuf, nstore, x, y0, slab, [&](int j, uint32_t& w0, uint32_t& w1, uint32_t& w2, uint32_t& w3) {
                const int i = b * 64 + j * 8;
                __nv_bfloat162 p0 = __floats2bfloat162_rn(v[i + 0], v[i + 1]);
                __nv_bfloat162 p1 = __floats2bfloat162_rn(v[i + 2], v[i + 3]);
                __nv_bfloat162 p2 = __floats2bfloat162_rn(v[i + 4], v[i + 5]);
                __nv_bfloat162 p3 = __floats2bfloat162_rn(v[i + 6], v[i + 7]);
                w0 = *reinterpret_cast<uint32_t*>(&p0);
                w1 = *reinterpret_cast<uint32_t*>(&p1);
                w2 = *reinterpret_cast<uint32_t*>(&p2);
                w3 = *reinterpret_cast<uint32_t*>(&p3);
            });
        }
    } else {
#pragma unroll
        for (int b = 0; b < kCols / 32; ++b) {
            const int32_t x = x0 + b * 32;
            if (x >= a.N) break;
            store_box(tmC, staging, nbuf, nstore, x, y0, slab, [&](int j, uint32_t& w0, uint32_t& w1, uint32_t& w2, uint32_t& w3) {
                const int i = b * 32 + j * 4;
                w0 = __float_as_uint(v[i + 0]);
                w1 = __float_as_uint(v[i + 1]);
                w2 = __float_as_uint(v[i + 2]);
                w3 = __float_as_uint(v[i + 3]);
            });
        }
    }
}

// v (+)= kPassCols columns (chunks c0, c0 + 1, ...) of this warp's block of a partial slot;
// kZero clears what it read (the atomic slot re-arms itself).
template <bool kAdd, bool kZero>
__device__ __forceinline__ void load_partial(float (&v)[kPassCols], float* blk, int c0, int lane) {
#pragma unroll
    for (int c = 0; c < kPassCols / 32; ++c)
#pragma unroll
        for (int q = 0; q < 8; ++q) {
            const int i = c * 32 + q * 4;
            float* p = blk + slot_f4(c0 + c, q, lane);
            const float4 x = ld_cg_f4(p);
            if (kAdd) {
                v[i] += x.x;
                v[i + 1] += x.y;
                v[i + 2] += x.z;
                v[i + 3] += x.w;
            } else {
                v[i] = x.x;
                v[i + 1] = x.y;
                v[i + 2] = x.z;
                v[i + 3] = x.w;
            }
            if (kZero) st_cg_f4(p, make_float4(0.f, 0.f, 0.f, 0.f));
        }
}

// Columns [o, o + 64) of one accumulator row (held in t) into the debug dump at d.
template <int kN>
__device__ __forceinline__ void dump_row(float* d, const uint32_t (&t)[kN], int o) {
#pragma unroll
    for (int q = 0; q < 16; ++q)
        *reinterpret_cast<float4*>(d + 4 * q) =
            make_float4(__uint_as_float(t[o + 4 * q]), __uint_as_float(t[o + 4 * q + 1]),
                        __uint_as_float(t[o + 4 * q + 2]), __uint_as_float(t[o + 4 * q + 3]));
}

// Epilogue state of one group of four warps (128 threads, one TMEM lane quadrant each), shared
// by the segments of one unit that the group takes.
template <int kCG, int kBN, int kGroup>
struct Epi {
    using S = Shape<kCG, kBN>;
    // The group's named barrier (barrier 2 is the TMEM hand-off), and, with two groups, the
    // accumulator every segment of this group uses.
    static constexpr uint32_t kBar = kGroup == 0 ? 1u : 3u;
    static constexpr bool kFixedBuf = kEpiGroups == 2;
    const KArgs& a;
    const CUtensorMap* tmC;
    const CUtensorMap* tmD;
    const Smem<S>& sm;
    uint32_t tmem_base;
    uint64_t deadline;
    volatile int* abort_flag;
    int lane, gt, quad, row;     // gt: thread index within the group
    int32_t r;                   // rank in the MMA pair: this CTA's rows are r * 128 .. of the tile
    int cta;                     // CTA within the tile: its block of a partial slot, its flags
    uint32_t tcol, staging, nstore;
    uint32_t nbuf;               // staging buffers in turn: kBoxes, or more in the ring (see `wide`)
    uint32_t ring;               // this warp's quarter of the ring (free once the unit's MAC loop is over)
    uint32_t pbar;               // this warp's two partial-load barriers, and their phase bits
    uint32_t pph;
    int ew;                      // index among the epilogue warps
    int* prefetch;               // shared hand-off word of the producer warp's partial copies
    volatile int* shared_tmp;    // shared word for the group's copy of an atomic result
    uint32_t tempty0, tempty1;   // accumulator-empty barriers (in the leader CTA)
    int64_t blk_off;
    int buf;                     // accumulator of the next segment (one group), and the phase parities
    uint32_t uses0, uses1;
    volatile int* last_flag;     // shared word: this group took a tile's last slab

    __device__ __forceinline__ float* block(int32_t slot) const {
        return a.slots + static_cast<int64_t>(slot * a.sch.cg + cta) * S::kCtaSlotFloats + blk_off;
    }

    // Split-K slabs, last arriver: this CTA's rows of tile g.tile in C = P[0] + P[1] + ...
    // + P[splits-1], summed left to right in FP32.
    __device__ __forceinline__ void reduce_slabs(const Seg& g) {
        int32_t trow, tcolumn;
        tile_coords(a.sch, g.tile, &trow, &tcolumn);
        const int32_t m0 = trow * (kCtaRows * kCG) + r * kCtaRows;
        const int32_t n0 = tcolumn * a.sch.tile_n;
        const int32_t gr = m0 + row;
        const int64_t slab = static_cast<int64_t>(a.M) * a.N;
#pragma unroll 1
        for (int p = 0; p < S::kPasses; ++p) {
            const int32_t c0 = n0 + p * kPassCols;
            float v[kPassCols];
#pragma unroll
            for (int i = 0; i < kPassCols; ++i) v[i] = 0.f;
            if (gr < a.M) {
                const float* rowp = a.slabs + static_cast<int64_t>(gr) * a.N + c0;
#pragma unroll
                for (int q = 0; q < kPassCols / 4; ++q) {
                    if (c0 + 4 * q < a.N) {
                        const float4 x = ld_cg_f4(rowp + 4 * q);
                        v[4 * q] = x.x;
                        v[4 * q + 1] = x.y;
                        v[4 * q + 2] = x.z;
                        v[4 * q + 3] = x.w;
                    }
                }
#pragma unroll 1
                for (int32_t j = 1; j < a.sch.splits; ++j) {
#pragma unroll
                    for (int q = 0; q < kPassCols / 4; ++q) {
                        if (c0 + 4 * q < a.N) {
                            const float4 x = ld_cg_f4(rowp + j * slab + 4 * q);
                            v[4 * q] += x.x;
                            v[4 * q + 1] += x.y;
                            v[4 * q + 2] += x.z;
                            v[4 * q + 3] += x.w;
                        }
                    }
                }
            }
            store_slice<kPassCols>(a, tmD, staging, nbuf, nstore, v, c0, m0 + quad * 32, -1);
        }
    }

    // One 4-column group of C (row gr, columns gc .. gc + 3) from its FP32 sum.
    __device__ __forceinline__ void store_c4(int32_t gr, int32_t gc, const float4& acc) const {
        const int64_t off = static_cast<int64_t>(gr) * a.N + gc;
        if (a.c_bf16) {
            __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x, acc.y);
            __nv_bfloat162 hi = __floats2bfloat162_rn(acc.z, acc.w);
            uint2 pk;
            pk.x = *reinterpret_cast<uint32_t*>(&lo);
            pk.y = *reinterpret_cast<uint32_t*>(&hi);
            *reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(a.C) + off) = pk;
        } else {
            *reinterpret_cast<float4*>(static_cast<float*>(a.C) + off) = acc;
        }
    }

    // Split-K slabs, shared sum: split g.slot's share of this CTA's 128 rows of tile g.tile,
    // rows [j * R, (j + 1) * R) with R = ceil(128 / splits), summed over the slabs in split
    // order (the reduction pass's order) and stored to C. The MAC loop is over (this is the
    // CTA's only work item), so the ring is idle: each epilogue warp takes every fourth row of
    // the share and brings that row's kBN columns from every slab into its quarter of the
    // ring with one bulk copy per (row, slab), all in flight at once, then sums them from
    // shared memory. A sum through registers would be bound by load latency (a thread can
    // keep only a few loads outstanding here). Returns false if a copy did not land in time.
    __device__ __forceinline__ bool reduce_slab_share(const Seg& g) {
        int32_t trow, tcolumn;
        tile_coords(a.sch, g.tile, &trow, &tcolumn);
        const int32_t rows_per = (kCtaRows + a.sch.splits - 1) / a.sch.splits;
        const int32_t r_begin = g.slot * rows_per;
        const int32_t r_end = imin(kCtaRows, r_begin + rows_per);
        const int32_t m0 = trow * (kCtaRows * kCG) + r * kCtaRows;
        const int32_t n0 = tcolumn * a.sch.tile_n;
        const int64_t slab = static_cast<int64_t>(a.M) * a.N;
        constexpr uint32_t kRowBytes = kBN * 4u;
        // Columns of the tile inside C: N % 8 == 0, so a row's copy is a multiple of 32 bytes,
        // and every source address (row * N + n0 floats) is 32-byte aligned.
        const int32_t cols = imin(kBN, a.N - n0);
        const int32_t rows_round = static_cast<int32_t>(kWarpRingBytes / (static_cast<uint32_t>(a.sch.splits) * kRowBytes));
        if (rows_round < 1) {
            reduce_slab_share_regs(m0, n0, r_begin, r_end, slab);
            return true;
        }
        const int wq = ew & 3;
        const uint32_t bar = pbar;  // this warp's first partial-load barrier
#pragma unroll 1
        for (int32_t r0 = r_begin + wq; r0 < r_end; r0 += 4 * rows_round) {
            const int32_t nr = imin(rows_round, (r_end - r0 + 3) / 4);  // rows r0, r0 + 4, ...
            if (lane == 0) {
                uint32_t bytes = 0;
                for (int32_t k = 0; k < nr; ++k)
                    if (m0 + r0 + 4 * k < a.M) bytes += static_cast<uint32_t>(a.sch.splits * cols) * 4u;
                fence_proxy_async_smem();  // this warp's earlier reads of the buffer come first
                mbar_arrive_expect_tx(bar, bytes);
                for (int32_t k = 0; k < nr; ++k) {
                    const int32_t gr = m0 + r0 + 4 * k;
                    if (gr >= a.M) continue;
                    const float* src = a.slabs + static_cast<int64_t>(gr) * a.N + n0;
                    for (int32_t j = 0; j < a.sch.splits; ++j)
                        bulk_load_g2s(ring + static_cast<uint32_t>(k * a.sch.splits + j) * kRowBytes, src + j * slab,
                                      static_cast<uint32_t>(cols) * 4u, bar);
                }
            }
            const uint32_t parity = pph & 1u;
            pph ^= 1u;
            if (!mbar_wait(bar, parity, abort_flag, deadline)) {
                (void)mbar_wait_until(bar, parity, globaltimer() + kDrainNs);  // let the copies land
                return false;
            }
            for (int32_t k = 0; k < nr; ++k) {
                const int32_t gr = m0 + r0 + 4 * k;
                if (gr >= a.M) continue;
                const uint32_t rowbuf = ring + static_cast<uint32_t>(k * a.sch.splits) * kRowBytes;
#pragma unroll 1
                for (int32_t c4 = lane; 4 * c4 < cols; c4 += 32) {
                    float4 acc = ld_shared_f4(rowbuf + 16u * c4);
#pragma unroll 4
                    for (int32_t j = 1; j < a.sch.splits; ++j) {
                        const float4 x = ld_shared_f4(rowbuf + static_cast<uint32_t>(j) * kRowBytes + 16u * c4);
                        acc.x += x.x;
                        acc.y += x.y;
                        acc.z += x.z;
                        acc.w += x.w;
                    }
                    store_c4(gr, n0 + 4 * c4, acc);
                }
            }
            __syncwarp();
        }
        return true;
    }

    // The shared sum through registers, for splits whose rows do not fit a ring quarter: work
    // items are (row, 4 columns), consecutive threads on consecutive columns of a row (512
    // contiguous bytes per warp load); an item's loads from all slabs go out 8 at a time.
    __device__ __forceinline__ void reduce_slab_share_regs(int32_t m0, int32_t n0, int32_t r_begin, int32_t r_end,
                                                           int64_t slab) {
        constexpr int kGroups = kBN / 4;  // 4-column groups per row
        constexpr int kBatch = 8;
        const int32_t items = (r_end > r_begin ? r_end - r_begin : 0) * kGroups;
#pragma unroll 1
        for (int32_t it = gt; it < items; it += kGroupThreads) {
            const int32_t gr = m0 + r_begin + it / kGroups;
            const int32_t gc = n0 + (it % kGroups) * 4;
            if (gr >= a.M || gc >= a.N) continue;  // N % 8 == 0: each group is all in or out
            const float* p = a.slabs + static_cast<int64_t>(gr) * a.N + gc;
            float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 1
            for (int32_t j0 = 0; j0 < a.sch.splits; j0 += kBatch) {
                float4 x[kBatch];
#pragma unroll
                for (int jj = 0; jj < kBatch; ++jj)
                    if (j0 + jj < a.sch.splits) x[jj] = ld_cg_f4(p + (j0 + jj) * slab);
#pragma unroll
                for (int jj = 0; jj < kBatch; ++jj) {
                    if (j0 + jj >= a.sch.splits) break;
                    if (j0 + jj == 0) {
                        acc = x[0];
                    } else {
                        acc.x += x[jj].x;
                        acc.y += x[jj].y;
                        acc.z += x[jj].z;
                        acc.w += x[jj].w;
                    }
                }
            }
            store_c4(gr, gc, acc);
        }
    }

    // The workspace indices a segment will use lie inside the extents the host sized.
    __device__ __forceinline__ bool in_bounds(const Seg& g) const {
        if (g.tile < 0 || g.tile >= a.sch.tiles) return false;
        if (g.role == kProducer) {
            const int32_t s = (a.atomic && !a.sch.sep) ? g.peer_begin : g.slot;
            return s >= 0 && s < a.sch.n_slots;
        }
        if (g.role == kOwner && a.sch.sep) return g.slot >= 0 && g.slot < a.sch.n_slots;
        if (g.role == kOwner)
            return g.peer_begin >= 0 && g.n_peers >= 1 && g.peer_begin + g.n_peers <= a.sch.n_slots;
        if (g.role == kSlab)
            return g.slot >= 0 && g.slot < a.sch.splits && (a.sch.partials != 2 || a.counters != nullptr);
        return true;
    }

    // Let this warp's partial copies still in flight (items waited .. issued - 1, all of them
    // started) land before the CTA may exit; bounded.
    __device__ __forceinline__ void drain_partials(int waited, int issued) {
        const uint64_t until = globaltimer() + kDrainNs;
        for (int j = waited; j < issued; ++j)
            (void)mbar_wait_until(pbar + 8u * static_cast<uint32_t>(j & 1), (pph >> (j & 1)) & 1u, until);
    }

    // One segment. kFixup: this segment is a split tile's owner and sums its peers' partials
    // here (without the separate fixup pass). `wide`: this is the unit's last segment, so once
    // its accumulator is complete the MAC loop is over and the ring is free. This warp's
    // quarter of the ring then stages all of its stores (12 buffers instead of kBoxes, so the
    // copies go out without waiting for a buffer). kBulk (a deterministic owner's last
    // segment, so also `wide`): the peers' partials come into the ring by bulk copies instead
    // of register loads. The producer warp, idle by then, has acquired the peers' flags and
    // started the first two copies as soon as the ring was free (run_producer); this warp
    // consumes them and issues the rest. `release`: a later segment of the unit will run in
    // this accumulator (the MMA issuer waits for it two segments on), so hand it back once
    // read; for the unit's last two segments nobody waits, and the group goes on unsynchronised.
    // Returns false when a wait gave up or a check failed (the caller stops).
    template <bool kFixup, bool kBulk>
    __device__ __forceinline__ bool segment(const Seg& g, uint64_t* tr, int seg, bool wide, bool release) {
        static_assert(kFixup || !kBulk, "bulk fetches are an owner's");
        constexpr int kChunks = kPassCols / 32;  // TMEM loads per pass
        constexpr bool bulk = kBulk;
        if (!in_bounds(g)) {  // same answer in every epilogue thread
            *abort_flag = 1;
            atomicCAS(a.status, 0, kErrBounds);
            return false;
        }
        // Where this CTA's rows of the tile go (computed before the accumulator waits).
        int32_t trow, tcolumn;
        tile_coords(a.sch, g.tile, &trow, &tcolumn);
        const int32_t m0 = trow * (kCtaRows * kCG) + r * kCtaRows;
        const int32_t n0 = tcolumn * a.sch.tile_n;
        const int32_t wy = m0 + quad * 32;  // first row of this warp's 32
        float* dump = a.dump ? a.dump +
                                   (static_cast<int64_t>(g.tile) * a.sch.iters + g.k_begin) *
                                       (static_cast<int64_t>(kCtaRows * kCG) * a.sch.tile_n) +
                                   static_cast<int64_t>(r * kCtaRows + row) * a.sch.tile_n
                             : nullptr;
        float v[kPassCols];
        if (kFixup && !bulk) {
            // Wait for every peer (this CTA's share of the partials), then fetch the first pass
            // of the first partial (or of the atomic sum) while this segment's MAC loop is
            // still running.
            bool ok = true;
            if (a.atomic) {
                ok = wait_flag(a.flags + g.peer_begin * a.sch.cg + cta, g.n_peers, deadline, abort_flag);
            } else {
                for (int32_t pi = 0; pi < g.n_peers && ok; ++pi)
                    ok = wait_flag(a.flags + (g.peer_begin + pi) * a.sch.cg + cta, 1, deadline, abort_flag);
            }
            if (named_bar_or(kBar, kGroupThreads, !ok)) {
                record_timeout(a, abort_flag);
                return false;
            }
            if (a.atomic)
                load_partial<false, true>(v, block(g.peer_begin), 0, lane);
            else
                load_partial<false, false>(v, block(g.peer_begin), 0, lane);
        }
        const int b = kFixedBuf ? kGroup : buf;
        const bool got = mbar_wait(sm.tfull(b), b ? uses1 : uses0, abort_flag, deadline);
        if (named_bar_or(kBar, kGroupThreads, !got || *abort_flag != 0)) {
            if (!got) record_timeout(a, abort_flag);
            return false;
        }
        tc_fence_after();
        if (tr && seg < kTraceSegs) tr[4 + 4 * seg + 2] = globaltimer();
        // Ring quarter: [0, 2 kPartBytes) the two partial buffers of a bulk owner, then its
        // 4 staging buffers; otherwise 12 staging buffers. Stores of earlier segments still in
        // flight read the staging block after the ring, not these buffers.
        if (wide) {
            staging = bulk ? ring + 2 * kPartBytes : ring;
            nbuf = bulk ? 4u : 12u;
            nstore = 0;
        }
        const int n_items = bulk ? S::kPasses * g.n_peers : 0;
        // Numerical control (tests): every partial this segment hands on (a producer's
        // partial, a Split-K slab, an owner's slot of the separate pass) is stored as zeros,
        // with its flags and counters raised as usual.
        const bool zero_store = a.zero_partials != 0 &&
                                (g.role == kProducer || g.role == kSlab || (g.role == kOwner && a.sch.sep != 0));
        int issued = bulk ? (n_items > 1 ? 2 : 1) : 0;  // the producer warp's copies
        int waited = 0;
        bool failed = false;



#pragma unroll 1
        for (int p = 0; p < S::kPasses; ++p) {
            if (kFixup && p > 0 && !bulk) {
                if (a.atomic)
                    load_partial<false, true>(v, block(g.peer_begin), kChunks * p, lane);
                else
                    load_partial<false, false>(v, block(g.peer_begin), kChunks * p, lane);
            }
            // This pass of the segment's own accumulator: one TMEM load for the whole pass,
            // or for an owner 64 columns at a time added to the first partial (own + P1: the
            // first step of the k-order fold).
            const uint32_t taddr = tmem_base + tcol + static_cast<uint32_t>(b * kBN + p * kPassCols);
            if (kFixup && !bulk) {
#pragma unroll
                for (int h = 0; h < kPassCols / 64; ++h) {
                    uint32_t t[64];
                    tmem_ld_32x32b_x64_sync(taddr + static_cast<uint32_t>(h * 64), t);
#pragma unroll
                    for (int i = 0; i < 64; ++i) v[h * 64 + i] = __uint_as_float(t[i]) + v[h * 64 + i];
                    if (dump) dump_row<64>(dump + p * kPassCols + h * 64, t, 0);
                }
            } else {
                uint32_t t[kPassCols];
                tmem_ld_pass_sync(taddr, t);
#pragma unroll
                for (int i = 0; i < kPassCols; ++i) v[i] = __uint_as_float(t[i]);
                if (dump) {
#pragma unroll
                    for (int h = 0; h < kPassCols / 64; ++h) dump_row<kPassCols>(dump + p * kPassCols + h * 64, t, h * 64);
                }
                if (zero_store) {
#pragma unroll
                    for (int i = 0; i < kPassCols; ++i) v[i] = 0.f;
                }
            }
            if (p == S::kPasses - 1 && release) {
                // The whole accumulator has been read: hand it back to the MMA issuer. One
                // thread per CTA arrives, after the group's barrier, and it is one that issues
                // no bulk copies (a release arrive waits for its thread's copies in flight).
                tc_fence_before();
                named_bar_sync(kBar, kGroupThreads);
                if (gt == 1) {
                    if (kCG == 1)
                        mbar_arrive(b ? tempty1 : tempty0);
                    else
                        mbar_arrive_cluster(b ? tempty1 : tempty0);
                }
            }

            if (kFixup && bulk) {
                // Turnstile from the ring: own + P(first peer) + P(next) ..., in k order; each
                // pass of each peer is one bulk copy, two in flight. A failed wait skips the
                // rest (the group decides after the loop).
#pragma unroll 1
                for (int32_t pi = 0; pi < g.n_peers; ++pi) {
                    const int j = p * g.n_peers + pi;
                    const uint32_t bit = static_cast<uint32_t>(j & 1);
                    if (!failed) failed = !mbar_wait(pbar + 8u * bit, (pph >> bit) & 1u, abort_flag, deadline);
                    if (failed) continue;
                    pph ^= 1u << bit;
                    ++waited;
                    const uint32_t src = ring + bit * kPartBytes;
#pragma unroll
                    for (int c = 0; c < kChunks; ++c)
#pragma unroll
                        for (int q = 0; q < 8; ++q) {
                            const float4 x = ld_shared_f4(src + static_cast<uint32_t>(slot_f4(c, q, lane)) * 4u);
                            const int i = c * 32 + q * 4;
                            v[i] += x.x;
                            v[i + 1] += x.y;
                            v[i + 2] += x.z;
                            v[i + 3] += x.w;
                        }
                    __syncwarp();  // every lane has read buffer `bit` before it is refilled
                    if (j + 2 < n_items) {
                        if (lane == 0) {
                            // The lanes' reads of the buffer, and (through the barrier) the
                            // producer warp's flag acquires, before this copy.
                            fence_proxy_async_smem();
                            fence_proxy_async_global();
                            fetch_partial(a, sm, g, cta, ew, j + 2);
                        }
                        ++issued;
                    }
                }
                if (!failed) store_slice<kPassCols>(a, tmC, staging, nbuf, nstore, v, n0 + p * kPassCols, wy, -1);
            } else if (kFixup) {
                // Turnstile: the remaining peers' partials, in k order.
                if (!a.atomic) {
                    for (int32_t pi = 1; pi < g.n_peers; ++pi)
                        load_partial<true, false>(v, block(g.peer_begin + pi), kChunks * p, lane);
                }
                store_slice<kPassCols>(a, tmC, staging, nbuf, nstore, v, n0 + p * kPassCols, wy, -1);
            } else if (g.role == kProducer || g.role == sk::kOwner) {
                // A producer's partial; with the separate fixup pass, an owner's too. The
                // pass sums them in k order, so the reduction mode does not apply there.
                const bool atomic = a.atomic && !a.sch.sep;
                float* blk = block(atomic ? g.peer_begin : g.slot);
#pragma unroll
                for (int c = 0; c < kChunks; ++c) {
                    if (atomic) {
#pragma unroll
                        for (int q = 0; q < 8; ++q) {
                            const int i = c * 32 + q * 4;
                            red_add_v4_f32(blk + slot_f4(kChunks * p + c, q, lane), v[i], v[i + 1], v[i + 2], v[i + 3]);
                        }
                    } else {
                        // Straight from registers: each warp store covers 512 contiguous bytes of
                        // the slot, so no staging buffer (and no wait for one) is needed.
#pragma unroll
                        for (int q = 0; q < 8; ++q) {
                            const int i = c * 32 + q * 4;
                            st_cg_f4(blk + slot_f4(kChunks * p + c, q, lane), make_float4(v[i], v[i + 1], v[i + 2], v[i + 3]));
                        }
                    }
                }
            } else if (g.role == kSlab) {
                store_slice<kPassCols>(a, tmC, staging, nbuf, nstore, v, n0 + p * kPassCols, wy, g.slot);
            } else {
                store_slice<kPassCols>(a, tmC, staging, nbuf, nstore, v, n0 + p * kPassCols, wy, -1);
            }
        }
        if (b)
            uses1 ^= 1u;
        else
            uses0 ^= 1u;
        if (!kFixedBuf) buf ^= 1;
        if (bulk && named_bar_or(kBar, kGroupThreads, failed)) {
            // Close the hand-off. If the producer warp never started its copies it never will;
            // otherwise let this warp's copies in flight land before the CTA may exit.
            if (gt == 0) *shared_tmp = atomicCAS(prefetch, 0, kPrefetchClosed);
            named_bar_sync(kBar, kGroupThreads);
            if (*shared_tmp >= kPrefetchIssued) drain_partials(waited, issued);
            record_timeout(a, abort_flag);
            return false;
        }

        if (g.role == kSlab && a.sch.partials == 2) {
            // Split-K slab, summed inside this launch (aligned split with a per-tile arrival
            // counter, as in the docc StreamK rewrite): publish the slab and count the arrival
            // at the tile. When every split of the tile is running at once, the splits share
            // the sum; otherwise the split that arrives last sums the tile's slabs alone. Both
            // add in split order. With split_partials = 1 a separate pass does the sum.
            if (lane == 0) {
                bulk_wait_group_all();
                fence_proxy_async_global();
            }
            __syncwarp();
            named_bar_sync(kBar, kGroupThreads);
            int32_t* cnt = a.counters + g.tile * a.sch.cg + cta;
            if (a.sch.coop) {
                // Every split of the tile is running (one work item per unit): wait until all
                // have arrived, then each sums its share of the rows. The counter goes on to
                // 2 * splits as the shares finish; the last to finish resets it to zero (by
                // then every split has passed its wait).
                if (gt == 0 && !a.skip_signal) (void)atom_add_acq_rel_gpu(cnt, 1);
                const bool all = wait_flag(cnt, a.sch.splits, deadline, abort_flag);
                if (named_bar_or(kBar, kGroupThreads, !all)) {
                    record_timeout(a, abort_flag);
                    return false;
                }
                fence_proxy_async_global();  // the peers' slabs, acquired above, are read by bulk copies
                if (named_bar_or(kBar, kGroupThreads, !reduce_slab_share(g))) {
                    record_timeout(a, abort_flag);
                    return false;
                }
                if (gt == 0 && atom_add_acq_rel_gpu(cnt, 1) == static_cast<uint32_t>(2 * a.sch.splits - 1))
                    atomicExch(cnt, 0);
                return true;
            }
            if (gt == 0) *last_flag = atom_add_acq_rel_gpu(cnt, 1) == static_cast<uint32_t>(a.sch.splits - 1);
            named_bar_sync(kBar, kGroupThreads);
            if (*last_flag) {
                (void)ld_acquire_gpu(a.counters + g.tile * a.sch.cg + cta);
                reduce_slabs(g);
                named_bar_sync(kBar, kGroupThreads);
                if (gt == 0) a.counters[g.tile * a.sch.cg + cta] = 0;
            }
        } else if (g.role == kProducer && !a.sch.sep) {
            // Every epilogue thread's share is stored (st.global from registers, or red.add in
            // atomic mode): publish it. The group's barrier orders every thread's stores before
            // one thread's release at GPU scope (release is cumulative), so an owner that
            // acquires the flag sees the whole partial. With the separate fixup pass nobody
            // waits: the pass runs after this launch.
            named_bar_sync(kBar, kGroupThreads);
            if (gt == 0 && !a.skip_signal) {
                if (a.atomic)
                    red_release_add_gpu(a.flags + g.peer_begin * a.sch.cg + cta, 1);
                else
                    st_release_gpu(a.flags + g.slot * a.sch.cg + cta, 1);
            }
        } else if (kFixup) {
            // Every epilogue thread has read the partials: re-arm the flags / counter. (With
            // bulk fetches every copy had completed before its warp read it, and the group
            // barrier after the passes already has every thread past its reads.)
            if (!bulk) named_bar_sync(kBar, kGroupThreads);
            if (gt == 0) {
                if (a.atomic) {
                    a.flags[g.peer_begin * a.sch.cg + cta] = 0;
                } else {
                    for (int32_t pi = 0; pi < g.n_peers; ++pi) a.flags[(g.peer_begin + pi) * a.sch.cg + cta] = 0;
                }
            }
        }
        return true;
    }
};

template <int kCG, int kBN, int kGroup>
__device__ void run_epilogue_group(const KArgs& a, const CUtensorMap* tmC, const CUtensorMap* tmD,
                                   const Smem<Shape<kCG, kBN>>& sm, uint32_t tmem_base, int unit, const CtaPos& pos,
                                   uint64_t deadline, volatile int* abort_flag, volatile int* last_flag,
                                   int* prefetch, volatile int* shared_tmp) {
    using S = Shape<kCG, kBN>;
    const int warp = threadIdx.x >> 5;
    const int ew = warp - 2;                  // index among the epilogue warps
    Epi<kCG, kBN, kGroup> e{a, tmC, tmD, sm, tmem_base, deadline, abort_flag};
    e.last_flag = last_flag + kGroup;
    e.lane = threadIdx.x & 31;
    e.gt = (ew & 3) * 32 + e.lane;            // index within the group
    e.quad = warp & 3;                        // TMEM lanes this warp may read: 32*quad ..
    e.row = e.quad * 32 + e.lane;             // row of this CTA's part of the tile
    e.r = static_cast<int32_t>(pos.rank);
    e.cta = static_cast<int>(pos.rank);
    e.tcol = static_cast<uint32_t>(e.quad * 32) << 16;
    e.staging = sm.base + S::kStagingOff + static_cast<uint32_t>(ew * kBoxes) * 4096u;
    e.nstore = 0;
    e.nbuf = kBoxes;
    e.ring = sm.base + static_cast<uint32_t>(ew & 3) * kWarpRingBytes;
    e.pbar = sm.pload(ew, 0);
    e.pph = 0;
    e.ew = ew;
    e.prefetch = prefetch;
    e.shared_tmp = shared_tmp;
    // The accumulator-empty barriers live in the pair's leader CTA.
    const uint32_t leader = 0u;
    e.tempty0 = kCG == 1 ? sm.tempty(0) : mapa_shared(sm.tempty(0), leader);
    e.tempty1 = kCG == 1 ? sm.tempty(1) : mapa_shared(sm.tempty(1), leader);
    e.blk_off = static_cast<int64_t>(e.quad) * S::kWarpSlotFloats;
    e.buf = 0;
    e.uses0 = e.uses1 = 0u;
    uint64_t* tr = (a.trace && e.gt == 0) ? a.trace + static_cast<int64_t>(blockIdx.x) * kTraceWords : nullptr;
    Walk w;
    Seg g;
    int n_seg = 0;  // segments of this unit (a walk of integer steps, before the first wait)
    w.init(a.sch, unit);
    while (w.next(a.sch, g)) ++n_seg;
    w.init(a.sch, unit);
    int seg = 0;  // the unit's segment index; the MMA issuer puts segment i in accumulator i % 2
    while (w.next(a.sch, g)) {
        if (seg % kEpiGroups == kGroup) {
            // The unit's last segment stages through the ring. With two groups the other group
            // may still be storing through its own buffers; the wide staging is for one only.
            const bool wide = seg == n_seg - 1 && kEpiGroups == 1;
            const bool release = seg + 2 < n_seg;
            bool ok;
            if (g.role == kOwner && !a.sch.sep)
                ok = (wide && !a.atomic) ? e.template segment<true, true>(g, tr, seg, true, release)
                                         : e.template segment<true, false>(g, tr, seg, wide, release);
            else
                ok = e.template segment<false, false>(g, tr, seg, wide, release);
            if (!ok) break;
            if (tr && seg < kTraceSegs) tr[4 + 4 * seg + 3] = globaltimer();
        }
        ++seg;
    }
    if (kEpiGroups == 1 && seg < n_seg - 1) {
        // Stopped before the last segment: close the producer warp's hand-off, and if it has
        // already started copies into the ring, let them land (bounded) before the CTA exits.
        if (e.gt == 0) *shared_tmp = atomicCAS(prefetch, 0, kPrefetchClosed);
        named_bar_sync(1, kGroupThreads);
        const int k = *shared_tmp - kPrefetchIssued;
        const uint64_t until = globaltimer() + kDrainNs;
        for (int j = 0; j < k; ++j) (void)mbar_wait_until(e.pbar + 8u * static_cast<uint32_t>(j & 1), 0u, until);
    }
    // Every TMA store of this warp has read its staging buffer before the CTA may exit. The
    // writes need not have landed: the grid completes only once they have, and nothing in
    // this launch reads C (partials and slabs are waited for in full before their flags).
    if (e.lane == 0) bulk_wait_group_read<0>();
    __syncwarp();
    if (tr && kGroup == 0) tr[2] = static_cast<uint64_t>(seg);
}

// Epilogue warps: group 0 (warps 2-5) and, with two groups, group 1 (warps 6-9).
template <int kCG, int kBN>
__device__ void run_epilogue(const KArgs& a, const CUtensorMap* tmC, const CUtensorMap* tmD,
                             const Smem<Shape<kCG, kBN>>& sm, uint32_t tmem_base, int unit, const CtaPos& pos,
                             uint64_t deadline, volatile int* abort_flag, volatile int* last_flag, int* prefetch,
                             volatile int* shared_tmp) {
    if (kEpiGroups == 1 || (threadIdx.x >> 5) < 6)
        run_epilogue_group<kCG, kBN, 0>(a, tmC, tmD, sm, tmem_base, unit, pos, deadline, abort_flag, last_flag,
                                        prefetch, shared_tmp);
    else
        run_epilogue_group<kCG, kBN, 1>(a, tmC, tmD, sm, tmem_base, unit, pos, deadline, abort_flag, last_flag,
                                        prefetch, shared_tmp);
}

// --------------------------------------------------------------------------- kernel
// kCG CTAs per MMA and per work tile (1, or a pair with cta_group::2); kBN accumulator
// columns per CTA.
template <bool kNT, int kCG, int kBN>
__global__ void __launch_bounds__(kThreads, 1)
    sk_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const __grid_constant__ CUtensorMap tmC, const __grid_constant__ CUtensorMap tmD,
                   const KArgs args) {
    using S = Shape<kCG, kBN>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    Smem<S> sm{smem_u32(smem)};
    uint8_t* bars = smem + S::kSmemBarOff;
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(bars + kBarTmemHolder);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(bars + kBarAbort);
    volatile int* last_flag = reinterpret_cast<volatile int*>(bars + kBarLastFlag);  // one per group
    int* prefetch = reinterpret_cast<int*>(bars + kBarPrefetch);
    volatile int* shared_tmp = reinterpret_cast<volatile int*>(bars + kBarSharedTmp);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    constexpr int kTileCtas = kCG;
    const uint32_t crank = kCG == 2 ? cluster_ctarank() : 0u;
    const CtaPos pos{crank};
    const uint32_t rank = pos.rank;
    const int units = static_cast<int>(gridDim.x) / kTileCtas;
    const int cid = static_cast<int>(blockIdx.x) / kTileCtas;
    const int unit = args.reverse ? units - 1 - cid : cid;

    if (threadIdx.x == 0) {
        for (int s = 0; s < S::kStages; ++s) {
            mbar_init(sm.full(s), 1);
            mbar_init(sm.empty(s), 1);  // one commit by the MMA issuer
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(sm.tfull(b), 1);
            mbar_init(sm.tempty(b), kCG);  // one arrive per CTA of the group that read it
        }
        mbar_init(sm.done(), 1);
        mbar_init(sm.tready(), 1);
        for (int w = 0; w < kEpiWarps; ++w) {
            mbar_init(sm.pload(w, 0), 1);
            mbar_init(sm.pload(w, 1), 1);
        }
        *abort_flag = 0;
        *prefetch = 0;
        fence_mbar_init();
        prefetch_tmap(&tmA);
        prefetch_tmap(&tmB);
        prefetch_tmap(&tmC);
        prefetch_tmap(&tmD);
    }
    // Barriers are initialised (in every CTA of the cluster) before anyone signals them. TMEM
    // is allocated afterwards, while the producer's first loads are already in flight.
    if (kCG == 2)
        cluster_sync();
    else
        __syncthreads();

    // Everything above touches only this CTA's own shared memory and the kernel parameters,
    // so under an overlapped launch it runs while the previous kernel on the stream is
    // still finishing (as do the producer's L2 prefetches of its first loads). Every thread that reads or writes global memory (A, B, C, the
    // workspace, the debug buffers) first waits for that kernel; TMEM is allocated before
    // the wait. Every thread signals the next overlapped launch once it is past its wait, so
    // that launch may begin when all of this grid's CTAs are.
    uint32_t tmem_base = 0;
    uint64_t start_clk = 0;  // thread 0, traced launches: SM clock at the start stamp
    // The producer and the MMA issuer take their unit's first segment from the walk before the
    // wait for the previous kernel: the walk reads only the kernel's arguments, and its first
    // step (cold instruction and constant caches, integer divisions) costs about a microsecond.
    Walk walk;
    Seg first{};
    bool have_first = false;
    // With overlap = 2 the caller states that A and B are not written by the kernel before
    // this one on the stream: the producer and the MMA issuer then start their first two
    // segments without waiting for it (they touch only A, B, shared and tensor memory until
    // their own later wait). A traced launch waits as usual, since the trace is global memory.
    const bool early = args.sch.overlap == 2 && args.trace == nullptr;
    if (warp == 0) {
        if (lane == 0) {
            if (args.sch.overlap == 1) prefetch_first_loads<kNT, kCG, kBN>(args, &tmA, &tmB, unit, pos);
            walk.init(args.sch, unit);
            have_first = walk.next(args.sch, first);
        }
        if (!early) grid_dep_wait();
        grid_dep_launch();
        const uint64_t deadline = globaltimer() + args.timeout_ns;  // wait limits count from here
        if (lane == 0) {
            if (args.trace) {
                args.trace[static_cast<int64_t>(blockIdx.x) * kTraceWords] = globaltimer();
                start_clk = clock64();
            }
            run_producer<kNT, kCG, kBN>(args, &tmA, &tmB, sm, walk, first, have_first, pos, deadline, abort_flag,
                                        prefetch, early);
        }
        // Warps 0 and 1 reconverge before the exit barrier: a CTA barrier counts a warp once
        // any of its threads arrives, so all 32 lanes must arrive together.
        __syncwarp();
    } else if (warp == 1) {
        if (kCG == 1) {
            tmem_alloc(smem_u32(tmem_holder), S::kTmemCols);
            tmem_relinquish();
        } else {
            tmem_alloc_pair(smem_u32(tmem_holder), S::kTmemCols);
            tmem_relinquish_pair();
        }
        // Hand the address to the epilogue warps (named barrier 2: this warp + the epilogue)
        // and, in a pair, tell the leader's MMA issuer that the peer's TMEM is allocated (the
        // leader's own allocation precedes its MMAs in this warp's program order).
        tc_fence_before();
        named_bar_arrive(2, 32 + kEpiThreads);
        if (kCG == 2 && rank != 0 && lane == 0)
            mbar_arrive_cluster(mapa_shared(sm.tready(), 0u));
        __syncwarp();
        tc_fence_after();
        tmem_base = *reinterpret_cast<volatile uint32_t*>(tmem_holder);
        if (lane == 0 && rank == 0) {
            walk.init(args.sch, unit);
            have_first = walk.next(args.sch, first);
        }
        if (!early) grid_dep_wait();
        grid_dep_launch();
        const uint64_t deadline = globaltimer() + args.timeout_ns;
        if (lane == 0 && rank == 0)
            run_mma<kNT, kCG, kBN>(args, sm, tmem_base, walk, first, have_first, deadline, abort_flag, early);
        __syncwarp();
    } else {
        named_bar_sync(2, 32 + kEpiThreads);
        tc_fence_after();
        tmem_base = *reinterpret_cast<volatile uint32_t*>(tmem_holder);
        grid_dep_wait();
        grid_dep_launch();
        const uint64_t deadline = globaltimer() + args.timeout_ns;
        run_epilogue<kCG, kBN>(args, &tmC, &tmD, sm, tmem_base, unit, pos, deadline, abort_flag, last_flag, prefetch,
                               shared_tmp);
    }

    tc_fence_before();
    // No remote shared-memory operation is outstanding here: the accumulator-empty arrives
    // stop two segments before the end, and every load and commit into the other CTA has
    // been waited on. So the exit barrier needs no release ordering.
    if (kCG == 2)
        cluster_sync_relaxed();
    else
        __syncthreads();
    if (args.trace && threadIdx.x == 0) {
        args.trace[static_cast<int64_t>(blockIdx.x) * kTraceWords + 1] = globaltimer();
        args.trace[static_cast<int64_t>(blockIdx.x) * kTraceWords + 3] = static_cast<uint64_t>(clock64()) - start_clk;
    }
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        if (kCG == 1)
            tmem_dealloc(tmem_base, S::kTmemCols);
        else
            tmem_dealloc_pair(tmem_base, S::kTmemCols);
    }
}

// --------------------------------------------------------------------------- host side
// One-CTA shapes launch cooperatively (the launch fails unless every unit is resident at
// once). Pair shapes launch as clusters of 2 without that attribute: the host has checked
// that every pair fits on the device at once (cudaOccupancyMaxActiveClusters), and an
// owner only ever waits for producer segments that run first in their own units.
// An overlapped launch (sch.overlap) adds programmatic stream serialization and, for the
// one-CTA shapes, relies on the same host-side residency check instead of the cooperative
// attribute. Its CTAs can only start once every CTA of the previous overlapped grid is past
// its own wait (each issues grid_dep_launch there), and they hold SMs only where the
// previous kernel's CTAs have left; once that kernel completes, all of this grid fits.
template <bool kNT, int kCG, int kBN>
cudaError_t launch_shape(const CUtensorMap& tmA, const CUtensorMap& tmB, const CUtensorMap& tmC,
                         const CUtensorMap& tmD, const KArgs& a, cudaStream_t stream) {
    using S = Shape<kCG, kBN>;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(a.sch.workers * kCG), 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = S::kSmemBytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    int n = 0;
    if (a.sch.overlap) {
        attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[n].val.programmaticStreamSerializationAllowed = 1;
        ++n;
    } else if (kCG == 1) {
        attr[n].id = cudaLaunchAttributeCooperative;
        attr[n].val.cooperative = 1;
        ++n;
    }
    if (kCG == 2) {
        attr[n].id = cudaLaunchAttributeClusterDimension;
        attr[n].val.clusterDim.x = kCG;
        attr[n].val.clusterDim.y = 1;
        attr[n].val.clusterDim.z = 1;
        ++n;
    }
    cfg.attrs = attr;
    cfg.numAttrs = n;
    return cudaLaunchKernelEx(&cfg, sk_gemm_kernel<kNT, kCG, kBN>, tmA, tmB, tmC, tmD, a);
}

template <int kCG, int kBN>
cudaError_t prepare_shape(int num_sms, int* max_units) {
    using S = Shape<kCG, kBN>;
    cudaError_t e = cudaFuncSetAttribute(sk_gemm_kernel<false, kCG, kBN>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, S::kSmemBytes);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(sk_gemm_kernel<true, kCG, kBN>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             S::kSmemBytes);
    if (e != cudaSuccess) return e;
    if (kCG == 1) {
        int n0 = 0, n1 = 0;
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n0, sk_gemm_kernel<false, kCG, kBN>, kThreads,
                                                          S::kSmemBytes);
        if (e != cudaSuccess) return e;
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n1, sk_gemm_kernel<true, kCG, kBN>, kThreads,
                                                          S::kSmemBytes);
        if (e != cudaSuccess) return e;
        *max_units = (n0 < n1 ? n0 : n1) * num_sms;
        return cudaSuccess;
    }
    // Units are clusters of kCG CTAs: as many as can be resident at once.
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(kCG * (num_sms / kCG)), 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = S::kSmemBytes;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = kCG;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int c0 = 0, c1 = 0;
    e = cudaOccupancyMaxActiveClusters(&c0, sk_gemm_kernel<false, kCG, kBN>, &cfg);
    if (e != cudaSuccess) return e;
    e = cudaOccupancyMaxActiveClusters(&c1, sk_gemm_kernel<true, kCG, kBN>, &cfg);
    if (e != cudaSuccess) return e;
    *max_units = c0 < c1 ? c0 : c1;
    return cudaSuccess;
}

}  // namespace

cudaError_t prepare_device(int num_sms, int* max_units) {
    cudaError_t e = prepare_shape<1, 128>(num_sms, &max_units[0]);
    if (e == cudaSuccess) e = prepare_shape<2, 128>(num_sms, &max_units[1]);
    if (e == cudaSuccess) e = prepare_shape<2, 256>(num_sms, &max_units[2]);
    if (e == cudaSuccess) e = prepare_shape<1, 256>(num_sms, &max_units[3]);
    return e;
}

cudaError_t launch_gemm(const CUtensorMap& tmA, const CUtensorMap& tmB, const CUtensorMap& tmC,
                        const CUtensorMap& tmD, bool nt, const KArgs& a, cudaStream_t stream) {
    const int cg = a.sch.cg, bn = a.sch.tile_n;
#define SK_LAUNCH(CG, BN)                                                             \
    return nt ? launch_shape<true, CG, BN>(tmA, tmB, tmC, tmD, a, stream)            \
              : launch_shape<false, CG, BN>(tmA, tmB, tmC, tmD, a, stream)
    if (cg == 1 && bn == 128) SK_LAUNCH(1, 128);
    if (cg == 2 && bn == 128) SK_LAUNCH(2, 128);
    if (cg == 2 && bn == 256) SK_LAUNCH(2, 256);
    if (cg == 1 && bn == 256) SK_LAUNCH(1, 256);
#undef SK_LAUNCH
    return cudaErrorInvalidValue;
}


}  // namespace sk
