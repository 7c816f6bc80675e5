"""GPU parity: the CUDA path through the C ABI against the CPU oracle.

Every schedule (data-parallel, Split-K, Stream-K, hybrid), both reductions (deterministic
turnstile, FP32 atomics) and both layouts (NN, NT) on the workloads' shapes, at sizes that
span several tiles with ragged edges, and at the full workload sizes. Pass criteria per
result: max |err| <= 2e-2 * max(1, |ref|) and relative Frobenius error <= 5e-3 against the
FP64 oracle, for the whole matrix and for every 128 x 128 tile; integer-valued inputs must
match exactly; sentinels and guards as in the split-K report's protocol.
"""
import numpy as np
import pytest
import torch

import synth
from oracle import gemm as og
from oracle import schedule as osch

from . import gpu_util as U

pytestmark = pytest.mark.gpu

DET, ATOM = 0, 1


@pytest.fixture(scope="module")
def sk():
    import __graft_entry__ as ge
    ge.build()
    import gemm_work_decomposition_gb300 as pkg
    return pkg


@pytest.fixture(scope="module")
def dev():
    assert torch.cuda.is_available()
    return torch.device("cuda:0")


@pytest.fixture(scope="module")
def dev_sms(dev):
    return torch.cuda.get_device_properties(dev).multi_processor_count


def _run(sk, dev, w, sched, red, sms, ws=None, **debug):
    A_bits, B_bits = U.inputs(w)
    A, B = U.to_dev(A_bits, dev), U.to_dev(B_bits, dev)
    got, guards, ws, status = U.gemm(sk, A, B, w.M, w.N, w.K, w.layout, sched, red, sms, w.out, dev, ws, **debug)
    assert status == sk.SK_OK
    assert guards
    return got, ws


SCHEDULES = [
    ("dp", dict(mode=0)),
    ("splitk2", dict(mode=1, splits=2)),
    ("splitk3", dict(mode=1, splits=3)),
    ("streamk", dict(mode=2)),
    ("hybrid", dict(mode=3)),
    ("slabs2", dict(mode=1, splits=2, split_partials=1)),
    ("slabs2_last", dict(mode=1, splits=2, split_partials=2)),
    ("streamk_sep", dict(mode=2, split_partials=1)),
    ("hybrid_sep", dict(mode=3, split_partials=1)),
]


# --------------------------------------------------------------------------- toy
TILES = [0, 1, 2, 3]


@pytest.mark.parametrize("tile", TILES)
@pytest.mark.parametrize("red", [DET, ATOM])
@pytest.mark.parametrize("name,kw", SCHEDULES)
def test_toy(sk, dev, name, kw, red, tile):
    # 5 tiles x 4 k-iterations on 4 units (Mental model figure); the pair and wide tile
    # shapes run the same problem over their coarser grids.
    w = synth.TOY
    sched = sk.schedule(units=4, tile=tile, **kw)
    got, _ = _run(sk, dev, w, sched, red, 4)
    assert not np.any(got == U.SENTINEL)
    U.assert_close(got, U.reference(w), name)


# --------------------------------------------------------------------------- exact
@pytest.mark.parametrize("tile", TILES)
@pytest.mark.parametrize("layout", ["NN", "NT"])
@pytest.mark.parametrize("red", [DET, ATOM])
@pytest.mark.parametrize("sms", [3, 7, 152])
@pytest.mark.parametrize("name,kw", SCHEDULES)
def test_integer_exact(sk, dev, name, kw, red, sms, layout, tile):
    # Ragged in M, N and K (300 x 264 x 520: 3 x 3 tiles, 9 k-iterations, the last one
    # 8 deep); integer inputs in [-4, 4] keep every partial sum exact in FP32, so every
    # schedule and reduction must equal the oracle exactly.
    M, N, K = 300, 264, 520
    A_bits, B_bits = synth.small_int_inputs(M, N, K, layout, 17)
    A, B = U.to_dev(A_bits, dev), U.to_dev(B_bits, dev)
    ref = og.ref_gemm(A_bits, B_bits, layout)
    sched = sk.schedule(tile=tile, **kw)
    got, guards, _, status = U.gemm(sk, A, B, M, N, K, layout, sched, red, sms, "f32", dev)
    assert status == sk.SK_OK and guards
    assert np.array_equal(got, ref)
    # BF16 output: the exact value rounded once to nearest even.
    got16, guards, _, status = U.gemm(sk, A, B, M, N, K, layout, sched, red, sms, "bf16", dev)
    assert status == sk.SK_OK and guards
    want16 = torch.from_numpy(ref.astype(np.float32)).to(torch.bfloat16).float().numpy()
    assert np.array_equal(got16, want16.astype(np.float64))


# --------------------------------------------------------------------------- wave-quantized
@pytest.mark.parametrize("red", [DET, ATOM])
@pytest.mark.parametrize("name,kw,sms", [
    ("dp", dict(mode=0), 148), ("splitk2", dict(mode=1, splits=2), 148), ("streamk", dict(mode=2), 148),
    ("hybrid", dict(mode=3), 148), ("hybrid_dev", dict(mode=3), None), ("streamk_dev", dict(mode=2), None),
    ("dp_pair128", dict(mode=0, tile=1), 148), ("hybrid_pair128", dict(mode=3, tile=1), 148),
    ("streamk_pair128", dict(mode=2, tile=1), 148), ("splitk2_pair128", dict(mode=1, splits=2, tile=1), 148),
    ("hybrid_pair256", dict(mode=3, tile=2), 148), ("streamk_pair256", dict(mode=2, tile=2), None),
    ("hybrid_wide256", dict(mode=3, tile=3), 148), ("streamk_wide256", dict(mode=2, tile=3), 148),
    ("hybrid_sep", dict(mode=3, split_partials=1), 148),
    ("hybrid_pair256_sep", dict(mode=3, tile=2, split_partials=1), 148)])
def test_waveq_full(sk, dev, dev_sms, name, kw, sms, red):
    # 2048 x 2432 x 4096: 304 tiles = 2 waves + 8 on 148 SMs, BF16 out; full comparison.
    w = synth.WAVEQ
    got, _ = _run(sk, dev, w, sk.schedule(**kw), red, sms or dev_sms)
    U.assert_close(got, U.reference(w), name)


def test_waveq_atomic_equals_deterministic_two_contributors(sk, dev):
    # The hybrid plan splits each tile over at most 2 units; 0 + a + b = 0 + b + a, so the
    # atomic reduction gives the deterministic bits here (first page, Case 3).
    w = synth.WAVEQ
    sched = sk.schedule(3)
    m = sk.sk_plan(w.M, w.N, w.K, 148, sched)
    assert max(m[-sk.SK_MAP_TILE * int(m[2]) + 1::sk.SK_MAP_TILE]) == 2
    det, _ = _run(sk, dev, w, sched, DET, 148)
    atom, _ = _run(sk, dev, w, sched, ATOM, 148)
    assert np.array_equal(det, atom)


# --------------------------------------------------------------------------- small-M NT
@pytest.mark.parametrize("partials", [1, 2], ids=["pass", "last"])
@pytest.mark.parametrize("tile", TILES)
@pytest.mark.parametrize("w", [synth.SMALLM_96, synth.SMALLM_256], ids=["m96", "m256"])
@pytest.mark.parametrize("s", [2, 4, 8, 16])
def test_smallm_split_slabs(sk, dev, dev_sms, w, s, tile, partials):
    # [splits, M, N] FP32 slabs then their sum (split-K report, Contract): every slab
    # against FP64 dot products over its own K range, and the reduced C. partials = 1
    # reduces in a second pass, 2 in the last split to arrive at each tile.
    sched = sk.schedule(1, splits=s, split_partials=partials, tile=tile)
    got, (ws, _) = _run(sk, dev, w, sched, DET, dev_sms)
    A_bits, B_bits = U.inputs(w)
    P_ref = og.ref_split_partials(A_bits, B_bits, "NT", s)
    P = ws[sk.SK_WS_HEADER_BYTES:sk.SK_WS_HEADER_BYTES + 4 * s * w.M * w.N].view(torch.float32)
    P = P.cpu().numpy().astype(np.float64).reshape(s, w.M, w.N)
    for j in range(s):
        U.assert_close(P[j], P_ref[j], f"slab {j}")
        assert np.abs(P[j] - P_ref[j]).max() <= 1e-4 * max(1.0, np.abs(P_ref[j]).max())
    ref = U.reference(w)
    U.assert_close(got, ref, "reduced")
    # A row 0 = 0 -> C row 0 is exactly +0.
    assert np.all(got[0] == 0.0) and not np.any(np.signbit(got[0]))
    # The reduction sums the slabs left to right in FP32.
    fold = P[0].astype(np.float32)
    for j in range(1, s):
        fold = fold + P[j].astype(np.float32)
    assert np.array_equal(got, fold.astype(np.float64))
    # The per-tile arrival counters after the slabs are back at zero for the next launch.
    off = -(-(sk.SK_WS_HEADER_BYTES + 4 * s * w.M * w.N) // 256) * 256
    assert not torch.any(ws[off:] != 0)


@pytest.mark.parametrize("tile", TILES)
@pytest.mark.parametrize("w", [synth.SMALLM_96, synth.SMALLM_256], ids=["m96", "m256"])
@pytest.mark.parametrize("name,kw", [("streamk", dict(mode=2)), ("hybrid", dict(mode=3)),
                                     ("splitk4", dict(mode=1, splits=4)), ("dp", dict(mode=0)),
                                     ("streamk_sep", dict(mode=2, split_partials=1))])
@pytest.mark.parametrize("red", [DET, ATOM])
def test_smallm_fixup(sk, dev, w, name, kw, red, tile):
    got, _ = _run(sk, dev, w, sk.schedule(tile=tile, **kw), red, 148)
    ref = U.reference(w)
    U.assert_close(got, ref, name)
    assert np.all(got[0] == 0.0)
    assert np.abs(got - ref).max() <= 1e-4 * max(1.0, np.abs(ref).max())


@pytest.mark.parametrize("out", ["f32", "bf16"])
@pytest.mark.parametrize("s,partials", [(3, 1), (3, 2), (16, 2)], ids=["s3pass", "s3launch", "s16launch"])
@pytest.mark.parametrize("tile", TILES)
@pytest.mark.parametrize("M,N,K", [(1, 8, 4096), (127, 8, 8192), (129, 136, 1024), (200, 1000, 1000),
                                   (300, 520, 2048)])
def test_slab_edges(sk, dev, M, N, K, tile, s, partials, out):
    # Split-K slabs at ragged edges (rows past M and columns past N inside a tile), summed by
    # the reduction pass (split_partials 1) or inside the launch (2: shared among the splits
    # when every split of a tile is resident, else by the last to arrive). C is the FP32
    # left fold of the slabs, rounded once to the output type, bit for bit.
    if s > -(-K // 64):
        pytest.skip("more splits than k-iterations")
    w = synth.Workload("slab_edge", M, N, K, "NT", "normal", 7, out=out)
    sched = sk.schedule(1, splits=s, split_partials=partials, tile=tile)
    got, (ws, _) = _run(sk, dev, w, sched, DET, 152)
    U.assert_close(got, U.reference(w), f"slabs s={s} partials={partials}")
    P = ws[sk.SK_WS_HEADER_BYTES:sk.SK_WS_HEADER_BYTES + 4 * s * M * N].view(torch.float32).reshape(s, M, N)
    fold = P[0].clone()
    for j in range(1, s):
        fold = fold + P[j]
    want = fold if out == "f32" else fold.to(torch.bfloat16).float()
    assert np.array_equal(got, want.cpu().numpy().astype(np.float64))


# --------------------------------------------------------------------------- sweep
@pytest.mark.parametrize("tile", [0, 1, 2])
@pytest.mark.parametrize("m", [128, 640, 1152, 1536, 2560, 4096])
@pytest.mark.parametrize("name,kw", [("dp", dict(mode=0)), ("splitk2", dict(mode=1, splits=2)),
                                     ("splitk4", dict(mode=1, splits=4)), ("splitk_cutlass", dict(mode=1)),
                                     ("splitk2_slabs", dict(mode=1, splits=2, split_partials=1)),
                                     ("splitk4_slabs", dict(mode=1, splits=4, split_partials=1)),
                                     ("splitk2_slabs_1launch", dict(mode=1, splits=2, split_partials=2)),
                                     ("splitk4_slabs_1launch", dict(mode=1, splits=4, split_partials=2)),
                                     ("streamk", dict(mode=2)), ("hybrid", dict(mode=3))])
def test_sweep(sk, dev, m, name, kw, tile):
    # The tile-count sweep's schedules; "splitk_cutlass" takes its split count from the
    # CUTLASS page's factor heuristic (32 at M = 128, 1 from 2432 up on 148 SMs).
    w = synth.sweep(m)
    if name == "splitk_cutlass":
        kw = dict(kw, splits=min(sk.sk_split_k_slices(m, m, w.K, 148), -(-w.K // 64)))
    got, _ = _run(sk, dev, w, sk.schedule(tile=tile, **kw), DET, 148)
    A_bits, B_bits = U.inputs(w)
    rows = U.sample_rows(m, 32, seed=m)
    U.assert_close(got[rows], og.ref_rows(A_bits, B_bits, "NN", rows), name)


# --------------------------------------------------------------------------- large / long-K
@pytest.mark.parametrize("tile", [0, 1, 2])
@pytest.mark.parametrize("name,kw", [("hybrid", dict(mode=3)), ("streamk", dict(mode=2)),
                                     ("streamk_sep", dict(mode=2, split_partials=1)),
                                     ("splitk16_slabs", dict(mode=1, splits=16, split_partials=1)),
                                     ("splitk16_launch", dict(mode=1, splits=16, split_partials=2))])
def test_skinny_long_k(sk, dev, name, kw, tile):
    # 512 x 512 x 65536: 16 tiles x 1024 k-iterations, up to 11 contributors per tile
    # (4 tiles over 74 pairs with the 256 x 256 pair tile: about 19 per tile). Split-K in 16
    # slabs: the pair tile's 64 work items are all resident and share each tile's sum; the
    # 128 x 128 tile's 256 items are not, and the last split to arrive sums its tile.
    w = synth.SKINNY
    got, _ = _run(sk, dev, w, sk.schedule(tile=tile, **kw), DET, 148)
    U.assert_close(got, U.reference(w), name)


@pytest.mark.parametrize("tile", [0, 2])
def test_large_8192(sk, dev, dev_sms, tile):
    w = synth.LARGE
    got, _ = _run(sk, dev, w, sk.schedule(3, tile=tile), DET, dev_sms)
    A_bits, B_bits = U.inputs(w)
    rows = U.sample_rows(w.M, 24, seed=5)
    U.assert_close(got[rows], og.ref_rows(A_bits, B_bits, "NN", rows), "8192^3")


# --------------------------------------------------------------------------- determinism
@pytest.mark.parametrize("w,sched_kw,units", [
    (synth.WAVEQ, dict(mode=3), 148), (synth.SKINNY, dict(mode=2), 148),
    (synth.sweep(256), dict(mode=2), 40), (synth.WAVEQ, dict(mode=3, tile=1), 148),
    (synth.SKINNY, dict(mode=2, tile=2), 148), (synth.sweep(512), dict(mode=2, tile=1, units=20), 148),
    (synth.SKINNY, dict(mode=2, tile=2, split_partials=1), 148)])
def test_deterministic_repeatable(sk, dev, w, sched_kw, units):
    # Deterministic mode: bit-identical over 10 runs and under the reversed unit -> CTA
    # order (the first page's Case 3 varies arrival order through a unit permutation).
    sched = sk.schedule(**sched_kw)
    first, ws = _run(sk, dev, w, sched, DET, units)
    for i in range(9):
        again, ws = _run(sk, dev, w, sched, DET, units, ws=ws, reverse_units=i % 2)
        assert np.array_equal(first, again)


@pytest.mark.parametrize("sep", [0, 1], ids=["owner", "pass"])
@pytest.mark.parametrize("tile,units", [(0, 40), (1, 20), (2, 10), (3, 20)])
def test_turnstile_k_order(sk, dev, tile, units, sep):
    # FP32 output, Stream-K over many units on few tiles (several contributors a tile): C
    # must be the left fold, in k order, of every segment's own FP32 partial, whether the
    # owner sums in-kernel or the separate fixup pass does.
    w = synth.Workload("t512", 512, 512, 4096, "NN", "normal", 31, out="f32")
    sched = sk.schedule(2, units=units, tile=tile, split_partials=sep)
    plan = osch.build_plan(w.M, w.N, w.K, 148, osch.STREAMK, units=units, tile=tile)
    tm, tn = plan.tile_m, plan.tile_n
    dump = torch.zeros(plan.tiles * plan.iters * tm * tn, dtype=torch.float32, device=dev)
    got, _ = _run(sk, dev, w, sched, DET, 148, dump=dump)
    D = dump.cpu().numpy().reshape(plan.tiles, plan.iters, tm, tn)
    want = np.zeros((w.M, w.N), dtype=np.float32)
    most = 0
    for t in range(plan.tiles):
        segs = sorted((s for s in plan.segments() if s.tile == t), key=lambda s: s.k_begin)
        most = max(most, len(segs))
        acc = D[t, segs[0].k_begin].copy()
        for s in segs[1:]:
            acc = acc + D[t, s.k_begin]
        tr, tc = osch.tile_coords(plan, t)
        r0, c0 = tr * tm, tc * tn
        want[r0:r0 + tm, c0:c0 + tn] = acc[:min(tm, w.M - r0), :min(tn, w.N - c0)]
    assert most >= 4
    assert np.array_equal(got, want.astype(np.float64))
    U.assert_close(got, U.reference(w), "turnstile")


@pytest.mark.parametrize("w,kw,sms", [
    (synth.WAVEQ, dict(mode=3), 148), (synth.WAVEQ, dict(mode=3, tile=2), 148),
    (synth.SKINNY, dict(mode=2), 148), (synth.SKINNY, dict(mode=2, tile=2), 148),
    (synth.SKINNY, dict(mode=2, tile=3), 148), (synth.SMALLM_96, dict(mode=3), 148),
    (synth.sweep(640), dict(mode=2, tile=1, units=11), 148)], ids=lambda v: getattr(v, "name", str(v)))
def test_separate_pass_equals_owner_fixup(sk, dev, w, kw, sms):
    # The separate fixup pass sums a split tile's partials in the owner's turnstile order
    # (own, then peers in k order), so it reproduces the deterministic in-kernel fixup bit
    # for bit.
    owner, _ = _run(sk, dev, w, sk.schedule(**kw), DET, sms)
    sep, _ = _run(sk, dev, w, sk.schedule(split_partials=1, **kw), DET, sms)
    assert np.array_equal(owner, sep)


# --------------------------------------------------------------------------- rasterization
@pytest.mark.parametrize("raster,swizzle", [(0, 2), (0, 3), (1, 0), (1, 4), (0, 256)])
@pytest.mark.parametrize("name,kw", [("dp", dict(mode=0)), ("splitk3", dict(mode=1, splits=3)),
                                     ("streamk", dict(mode=2)), ("hybrid", dict(mode=3)),
                                     ("slabs2", dict(mode=1, splits=2, split_partials=1)),
                                     ("streamk_sep", dict(mode=2, split_partials=1))])
@pytest.mark.parametrize("tile", [0, 2])
def test_rasterized_tile_order(sk, dev, name, kw, raster, swizzle, tile):
    # A ragged 1000 x 1016 x 520 NT problem (8 x 8 tiles of 128, 4 x 4 of 256) in every tile
    # order: each tile lands where tile_coords puts it, edges clipped.
    w = synth.Workload("r", 1000, 1016, 520, "NT", "normal", 41, out="f32")
    got, _ = _run(sk, dev, w, sk.schedule(tile=tile, raster=raster, swizzle=swizzle, **kw), DET, 37)
    assert not np.any(got == U.SENTINEL)
    U.assert_close(got, U.reference(w), name)


@pytest.mark.parametrize("raster,swizzle", [(0, 4), (1, 8)])
def test_rasterized_waveq_and_large(sk, dev, raster, swizzle):
    w = synth.WAVEQ
    got, _ = _run(sk, dev, w, sk.schedule(3, tile=2, raster=raster, swizzle=swizzle), DET, 148)
    U.assert_close(got, U.reference(w), "waveq")
    w = synth.LARGE
    got, _ = _run(sk, dev, w, sk.schedule(0, tile=2, raster=raster, swizzle=swizzle), DET, 148)
    A_bits, B_bits = U.inputs(w)
    rows = U.sample_rows(w.M, 16, seed=raster * 10 + swizzle)
    U.assert_close(got[rows], og.ref_rows(A_bits, B_bits, "NN", rows), "8192^3")


# --------------------------------------------------------------------------- atomics
@pytest.mark.parametrize("tile", [0, 1, 2])
def test_atomic_many_contributors(sk, dev, tile):
    # Skinny shape, up to 11 contributors per tile: within tolerance. With three or more
    # contributors the FP32 additions follow the peers' finishing order, so the last bits
    # may differ from run to run (first page, Case 3).
    w = synth.SKINNY
    got, ws = _run(sk, dev, w, sk.schedule(2, tile=tile), ATOM, 148)
    U.assert_close(got, U.reference(w), "atomic")
    again, _ = _run(sk, dev, w, sk.schedule(2, tile=tile), ATOM, 148, ws=ws, reverse_units=1)
    U.assert_close(again, U.reference(w), "atomic reversed")


# --------------------------------------------------------------------------- edges
@pytest.mark.parametrize("M,N,K", [(1, 8, 8), (1, 8, 4096), (129, 136, 72), (128, 128, 8), (200, 1000, 1000),
                                   (127, 8, 65536 // 8)])
@pytest.mark.parametrize("tile", TILES)
@pytest.mark.parametrize("name,kw", [("dp", dict(mode=0)), ("streamk", dict(mode=2)), ("hybrid", dict(mode=3)),
                                     ("splitk", dict(mode=1, splits=1)),
                                     ("streamk_sep", dict(mode=2, split_partials=1))])
def test_edges(sk, dev, M, N, K, name, kw, tile):
    w = synth.Workload("e", M, N, K, "NT", "normal", 3, out="f32")
    got, _ = _run(sk, dev, w, sk.schedule(tile=tile, **kw), DET, 152)
    U.assert_close(got, U.reference(w), name)


def test_k_zero_and_empty(sk, dev):
    C = torch.full((16 * 8 + 64,), 7.0, device=dev)
    st = torch.cuda.current_stream(dev)
    sk.sk_gemm(0, 0, C, sk.SK_F32, 16, 8, 0, sk.SK_NN, sk.schedule(0), 0, 148, 0, 0, st)
    torch.cuda.synchronize()
    h = C.cpu().numpy()
    assert np.all(h[:128] == 0.0) and np.all(h[128:] == 7.0)
    sk.sk_gemm(0, 0, C, sk.SK_F32, 0, 8, 64, sk.SK_NN, sk.schedule(0), 0, 148, 0, 0, st)
    torch.cuda.synchronize()
    assert np.all(C.cpu().numpy()[:128] == 0.0)


def test_residency_limit(sk, dev, dev_sms):
    w = synth.sweep(4096)
    A = torch.zeros((8, 8), dtype=torch.bfloat16, device=dev)
    ws = torch.zeros(1 << 20, dtype=torch.uint8, device=dev)
    C = torch.zeros((4096, 4096), dtype=torch.float32, device=dev)
    with pytest.raises(sk.SkError) as e:
        sk.sk_gemm(A, A, C, sk.SK_F32, w.M, w.N, w.K, sk.SK_NN, sk.schedule(0), 0, dev_sms + 1, ws, 1 << 20)
    assert e.value.code == sk.SK_ERESIDENCY


# --------------------------------------------------------------------------- reduce pass
@pytest.mark.parametrize("s,mn,out", [(1, 4096, "f32"), (3, 1 << 20, "f32"), (16, 96 * 512, "bf16")])
def test_reduce_splits(sk, dev, s, mn, out):
    P = torch.randn(s * mn, dtype=torch.float32, generator=torch.Generator().manual_seed(s)).to(dev)
    dt = torch.float32 if out == "f32" else torch.bfloat16
    C = torch.full((mn + 64,), 11.0, dtype=dt, device=dev)
    sk.sk_reduce_splits(P, C, sk.SK_F32 if out == "f32" else sk.SK_BF16, s, mn, torch.cuda.current_stream(dev))
    torch.cuda.synchronize()
    h = P.cpu().numpy().reshape(s, mn)
    fold = h[0].copy()
    for j in range(1, s):
        fold = fold + h[j]
    want = torch.from_numpy(fold).to(dt).float().numpy()
    got = C.float().cpu().numpy()
    assert np.array_equal(got[:mn], want) and np.all(got[mn:] == 11.0)


# --------------------------------------------------------------------------- time-out
@pytest.mark.parametrize("red", [DET, ATOM])
@pytest.mark.parametrize("overlap", [0, 1])
@pytest.mark.parametrize("tile", [0, 1, 2])
def test_wait_timeout_reports_status(sk, dev, tile, overlap, red):
    # Producers store but never raise their flag: every owner's wait runs out after 50 ms,
    # the kernel unwinds and records SK_ETIMEOUT; the context stays usable and the
    # workspace works again once zeroed. Toy problem on 4 units: unit 0 ends with a 1-iteration
    # owner segment, so with the deterministic reduction its peers' partials go through the
    # producer warp's ring copies, and the time-out runs out in the producer warp's flag wait
    # and in the epilogue's copy wait (the hand-off word stays closed).
    w = synth.TOY
    sched = sk.schedule(2, units=4, tile=tile, overlap=overlap)
    A_bits, B_bits = U.inputs(w)
    A, B = U.to_dev(A_bits, dev), U.to_dev(B_bits, dev)
    ws = U.new_workspace(sk, w.M, w.N, w.K, 4, sched, red, dev)
    _, _, _, status = U.gemm(sk, A, B, w.M, w.N, w.K, "NN", sched, red, 4, "f32", dev, ws,
                             skip_producer_signal=1, timeout_ns=50_000_000)
    assert status == sk.SK_ETIMEOUT
    assert sk.sk_status(ws[0]) == sk.SK_OK
    ws[0].zero_()
    got, guards, _, status = U.gemm(sk, A, B, w.M, w.N, w.K, "NN", sched, red, 4, "f32", dev, ws)
    assert status == sk.SK_OK and guards
    U.assert_close(got, U.reference(w), "after time-out")


@pytest.mark.parametrize("s", [2, 8])
def test_shared_slab_wait_timeout(sk, dev, dev_sms, s):
    # Split-K slabs summed in the launch, every split on a unit of its own (small-M: 4 tiles
    # x s splits): the splits wait for each other before sharing the sum. With their
    # arrivals suppressed the wait runs out after 50 ms and the kernel records SK_ETIMEOUT;
    # the context stays usable and the workspace works again once zeroed.
    w = synth.SMALLM_96
    sched = sk.schedule(1, s, split_partials=2)
    A_bits, B_bits = U.inputs(w)
    A, B = U.to_dev(A_bits, dev), U.to_dev(B_bits, dev)
    ws = U.new_workspace(sk, w.M, w.N, w.K, dev_sms, sched, DET, dev)
    _, _, _, status = U.gemm(sk, A, B, w.M, w.N, w.K, "NT", sched, DET, dev_sms, "f32", dev, ws,
                             skip_producer_signal=1, timeout_ns=50_000_000)
    assert status == sk.SK_ETIMEOUT
    ws[0].zero_()
    got, guards, _, status = U.gemm(sk, A, B, w.M, w.N, w.K, "NT", sched, DET, dev_sms, "f32", dev, ws)
    assert status == sk.SK_OK and guards
    U.assert_close(got, U.reference(w), "after time-out")


# --------------------------------------------------------------------------- page, Case 3 claims
def test_case3_interpreter_claims(sk, dev):
    # The first page's Case 3 run, at its structure with this library's tiles: 16 tiles x 32
    # k-iterations (512 x 512 x 2048 with 128 x 128 x 64), Stream-K on 12 and on 40 units,
    # FP32 output. Claims: Stream-K and data-parallel are both within tolerance but not the
    # same bits; a fixed-order fixup does not change under reversed unit order (nor between
    # the owner's in-kernel fixup and the separate fixup pass); atomics with at most 2
    # contributors per tile equal the fixed-order bits. With up to 4 contributors, atomics
    # may differ from run to run: only the tolerance is required there.
    w = synth.Workload("case3", 512, 512, 2048, "NN", "normal", 33, out="f32")
    ref = U.reference(w)
    dp, _ = _run(sk, dev, w, sk.schedule(0), DET, 16)
    sk12, ws12 = _run(sk, dev, w, sk.schedule(2, units=12), DET, 148)
    U.assert_close(dp, ref, "dp")
    U.assert_close(sk12, ref, "streamk 12")
    assert np.count_nonzero(dp != sk12) > 0
    rev12, _ = _run(sk, dev, w, sk.schedule(2, units=12), DET, 148, reverse_units=1)
    assert np.array_equal(sk12, rev12)
    at12, _ = _run(sk, dev, w, sk.schedule(2, units=12), ATOM, 148, reverse_units=1)
    assert np.array_equal(sk12, at12)
    plan40 = osch.build_plan(w.M, w.N, w.K, 148, osch.STREAMK, units=40)
    assert max(c for _, c in osch.tile_rows(plan40)) == 4
    own40, _ = _run(sk, dev, w, sk.schedule(2, units=40), DET, 148)
    rev40, _ = _run(sk, dev, w, sk.schedule(2, units=40, split_partials=1), DET, 148, reverse_units=1)
    assert np.array_equal(own40, rev40)
    at40, _ = _run(sk, dev, w, sk.schedule(2, units=40), ATOM, 148, reverse_units=1)
    U.assert_close(at40, ref, "atomic 40")


# --------------------------------------------------------------------------- trace record
@pytest.mark.parametrize("tile,nsms", [(0, 148), (2, 148), (1, 148), (3, 148)])
def test_trace_record(sk, dev, tile, nsms):
    # The per-CTA trace (sk_debug_opts.trace) of the hybrid rule on the wave-quantized GEMM,
    # checked against the plan map: every CTA walks its unit's segments; start <= end; for
    # each traced segment the MMA leader's first issue <= last commit, and the epilogue takes
    # the accumulator after that commit and finishes after it takes it; word 3 counts the SM
    # cycles between start and end, a clock between 0.5 and 3 GHz. The GEMM's result is still
    # the oracle's.
    w = synth.WAVEQ
    sched = sk.schedule(3, tile=tile)
    plan = sk.sk_plan(w.M, w.N, w.K, nsms, sched)
    cg, workers = int(plan[14]), int(plan[4])
    ncta = workers * cg
    segs = {}
    for i in range(int(plan[7])):
        r = plan[sk.SK_MAP_HEADER + sk.SK_MAP_SEG * i: sk.SK_MAP_HEADER + sk.SK_MAP_SEG * (i + 1)]
        segs[int(r[0])] = segs.get(int(r[0]), 0) + 1
    tr = torch.zeros(ncta * sk.SK_TRACE_WORDS, dtype=torch.int64, device=dev)
    got, _ = _run(sk, dev, w, sched, DET, nsms, trace=tr)
    U.assert_close(got, U.reference(w), "traced")
    T = tr.cpu().numpy().reshape(ncta, sk.SK_TRACE_WORDS).astype(np.int64)
    for c in range(ncta):
        unit, rank_in_pair = c // cg, (c % cg) % 2
        n = segs.get(unit, 0)
        assert T[c, 2] == n, (c, T[c, 2], n)
        assert 0 < T[c, 0] <= T[c, 1]
        mhz = T[c, 3] / max(1, T[c, 1] - T[c, 0]) * 1e3
        assert 500 <= mhz <= 3000, (c, mhz)
        for s in range(min(n, sk.SK_TRACE_SEGS)):
            issue, commit, acc, done = T[c, 4 + 4 * s: 8 + 4 * s]
            assert T[c, 0] <= acc <= done <= T[c, 1] + 10_000, (c, s)
            if rank_in_pair == 0:  # the MMA stamps come from the leader of each MMA pair
                assert T[c, 0] <= issue <= commit <= acc + 10_000, (c, s)


# --------------------------------------------------------------------------- numerical control
CONTROL_CASES = [
    # (id, workload, schedule, reduction, units)
    ("toy_streamk", synth.TOY, dict(mode=2, units=4), DET, 4),
    ("toy_streamk_atomic", synth.TOY, dict(mode=2, units=4), ATOM, 4),
    ("waveq_hybrid_pair", synth.WAVEQ, dict(mode=3, tile=2), DET, 148),
    ("waveq_hybrid_sep", synth.WAVEQ, dict(mode=3, tile=2, split_partials=1), DET, 148),
    ("skinny_streamk", synth.SKINNY, dict(mode=2, tile=0), DET, 148),
    ("smallm96_slabs8", synth.SMALLM_96, dict(mode=1, splits=8, split_partials=1), DET, 148),
    ("smallm256_slabs4_last", synth.SMALLM_256, dict(mode=1, splits=4, split_partials=2), DET, 148),
]


@pytest.mark.parametrize("name,w,kw,red,sms", CONTROL_CASES, ids=[c[0] for c in CONTROL_CASES])
def test_zeroed_partials_fail_the_checks(sk, dev, name, w, kw, red, sms):
    # Numerical control ("Consecutive-B split-K NAX GEMM", Contract and numerical coverage):
    # with every partial store zeroed on the GPU (flags still raised), the same parity check
    # that passes on the real result must fail. Sampled rows keep the full-size cases quick.
    sched = sk.schedule(**kw)
    A_bits, B_bits = U.inputs(w)
    rows = U.sample_rows(w.M, 24, seed=7)
    ref = og.ref_rows(A_bits, B_bits, w.layout, rows)
    good, _ = _run(sk, dev, w, sched, red, sms)
    U.assert_close(good[rows], ref, name)
    bad, _ = _run(sk, dev, w, sched, red, sms, zero_partials=1)
    with pytest.raises(AssertionError):
        U.assert_close(bad[rows], ref, name + " (zeroed partials)")
    # Only the handed-on partials changed: tiles no unit split are still right.
    m = sk.sk_plan(w.M, w.N, w.K, sms, sched)
    tiles = int(m[2])
    trows = m[len(m) - sk.SK_MAP_TILE * tiles:].reshape(tiles, sk.SK_MAP_TILE)
    tm, tn = int(m[12]), int(m[13])
    for t in range(tiles):
        if int(trows[t, 1]) == 1 and not kw.get("split_partials"):
            r, c = int(trows[t, 2]) * tm, int(trows[t, 3]) * tn
            assert np.array_equal(bad[r:r + tm, c:c + tn], good[r:r + tm, c:c + tn])


# --------------------------------------------------------------------------- Stream-K groups
GROUP_CASES = [
    # (id, workload, schedule, units)
    ("toy_g2", synth.TOY, dict(mode=2, units=4, sk_groups=2), 4),
    ("toy_g2_sep", synth.TOY, dict(mode=2, units=4, sk_groups=2, split_partials=1), 4),
    ("skinny_g8", synth.SKINNY, dict(mode=2, sk_groups=8), 148),
    ("skinny_pair_g4_sep", synth.SKINNY, dict(mode=2, tile=2, sk_groups=4, split_partials=1), 148),
    ("waveq_hybrid_g8", synth.WAVEQ, dict(mode=3, sk_groups=8), 148),
    ("waveq_hybrid_pair_g8", synth.WAVEQ, dict(mode=3, tile=2, sk_groups=8), 148),
    ("large_streamk_pair_g8", synth.LARGE, dict(mode=2, tile=2, sk_groups=8), 148),
]


@pytest.mark.parametrize("red", [DET, ATOM])
@pytest.mark.parametrize("name,w,kw,sms", GROUP_CASES, ids=[c[0] for c in GROUP_CASES])
def test_streamk_groups(sk, dev, name, w, kw, sms, red):
    # max_sk_groups_ grouping (first page, Case 4 knob table): the grouped plan (planner ==
    # oracle on the host) runs to the oracle's result; deterministic runs are bit-identical
    # under reversed unit order, and the map uses more than one group.
    sched = sk.schedule(**kw)
    plan = sk.sk_plan(w.M, w.N, w.K, sms, sched)
    assert int(plan[17]) >= 2
    got, _ = _run(sk, dev, w, sched, red, sms)
    A_bits, B_bits = U.inputs(w)
    if w.M * w.N <= 2048 * 2432:
        U.assert_close(got, U.reference(w), name)
    else:
        rows = U.sample_rows(w.M, 16, seed=3)
        U.assert_close(got[rows], og.ref_rows(A_bits, B_bits, w.layout, rows), name)
    if red == DET:
        rev, _ = _run(sk, dev, w, sched, DET, sms, reverse_units=1)
        assert np.array_equal(got, rev)
