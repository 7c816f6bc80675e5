"""Overlapped launches (sk_schedule.overlap = 1: programmatic dependent launch) against the
same calls launched without overlap. Each overlapped kernel sets up while the kernel
before it on the stream finishes, and must wait for it before touching global memory, so
every result must equal the non-overlapped one bit for bit:
  - chains where each GEMM reads the output of the GEMM just before it;
  - inputs rewritten by a PyTorch kernel right before each GEMM;
  - back-to-back calls with different inputs that share one workspace (turnstile flags,
    slab arrival counters, atomic tiles and fixup slots carried from call to call).
With overlap = 2 (A and B not written by the kernel before) the first two segments' loads
and MMAs may also run before that kernel completes; C, the workspace and the flags may
not, so back-to-back calls over independent operands, sharing one workspace or one C,
must give the same bits as well, and wait limits must not run out while a long kernel
ahead is still running.
"""
import numpy as np
import pytest
import torch

import synth

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


SCHEDULES = [
    ("dp", dict(mode=0)),
    ("splitk3", dict(mode=1, splits=3)),
    ("streamk", dict(mode=2)),
    ("hybrid", dict(mode=3)),
    ("slabs2", dict(mode=1, splits=2, split_partials=1)),
    ("slabs3_one_launch", dict(mode=1, splits=3, split_partials=2)),
    ("streamk_sep", dict(mode=2, split_partials=1)),
]


def _bf16(bits, dev):
    return U.to_dev(bits, dev)


def _chain(sk, dev, X0, Ws, M, K, kw, overlap, sms):
    """X_{i+1} = X_i . W_i (NN, BF16 out) for every W_i, all launched back to back."""
    sched = sk.schedule(overlap=overlap, **kw)
    nbytes = sk.sk_workspace_size(M, K, K, sms, sched, DET)
    ws = torch.zeros(nbytes, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    xs = [X0]
    # Every output starts as a sentinel so that a read ahead of its producer shows.
    outs = [torch.full((M, K), U.SENTINEL, dtype=torch.bfloat16, device=dev) for _ in Ws]
    torch.cuda.synchronize(dev)
    for W, Y in zip(Ws, outs):
        sk.sk_gemm(xs[-1], W, Y, sk.SK_BF16, M, K, K, sk.SK_NN, sched, DET, sms, ws, nbytes, stream)
        xs.append(Y)
    assert sk.sk_status(ws, stream) == sk.SK_OK
    return [y.float().cpu().numpy() for y in outs]


@pytest.mark.parametrize("tile", [0, 2])
@pytest.mark.parametrize("name,kw", SCHEDULES)
def test_overlapped_chain_equals_serial(sk, dev, name, kw, tile):
    # 640 x 768 x 768 (ragged in M for both tile shapes), five dependent GEMMs: the grids
    # are small enough that an overlapped GEMM's CTAs all fit beside the running one, so a
    # missing wait would read its input before it is written.
    M, K = 640, 768
    X0 = _bf16(synth.make_inputs(synth.Workload("chain_x", M, K, K, seed=40))[0], dev)
    Ws = [_bf16(synth.make_inputs(synth.Workload("chain_w", K, K, K, seed=41 + i))[1], dev) for i in range(5)]
    kw = dict(kw, tile=tile)
    ref = _chain(sk, dev, X0, Ws, M, K, kw, 0, 148)
    got = _chain(sk, dev, X0, Ws, M, K, kw, 1, 148)
    for i, (g, r) in enumerate(zip(got, ref)):
        assert not np.any(r == U.SENTINEL)
        assert np.array_equal(g, r), (name, tile, i)


@pytest.mark.parametrize("tile", [0, 2])
def test_overlapped_after_torch_kernel(sk, dev, tile):
    # A PyTorch elementwise kernel rewrites A right before each overlapped GEMM; each GEMM
    # must see that step's A.
    M, N, K = 512, 640, 1024
    srcs = [_bf16(synth.make_inputs(synth.Workload("torch_a", M, N, K, seed=50 + i))[0], dev) for i in range(6)]
    B = _bf16(synth.make_inputs(synth.Workload("torch_b", M, N, K, seed=49))[1], dev)
    A = torch.empty_like(srcs[0])
    stream = torch.cuda.current_stream(dev)

    def run(overlap):
        sched = sk.schedule(mode=3, tile=tile, overlap=overlap)
        nbytes = sk.sk_workspace_size(M, N, K, 148, sched, DET)
        ws = torch.zeros(nbytes, dtype=torch.uint8, device=dev)
        C = torch.empty((M, N), dtype=torch.float32, device=dev)
        outs = []
        for s in srcs:
            torch.mul(s, 1.0, out=A)
            sk.sk_gemm(A, B, C, sk.SK_F32, M, N, K, sk.SK_NN, sched, DET, 148, ws, nbytes, stream)
            outs.append(C.clone())
        assert sk.sk_status(ws, stream) == sk.SK_OK
        return [o.cpu().numpy() for o in outs]

    ref, got = run(0), run(1)
    for i, (g, r) in enumerate(zip(got, ref)):
        assert np.array_equal(g, r), i
    assert not np.array_equal(ref[0], ref[1])


@pytest.mark.parametrize("red", [DET, ATOM])
@pytest.mark.parametrize("tile", [0, 2])
@pytest.mark.parametrize("name,kw", [("streamk", dict(mode=2)), ("hybrid", dict(mode=3)),
                                     ("slabs3_one_launch", dict(mode=1, splits=3, split_partials=2)),
                                     ("streamk_sep", dict(mode=2, split_partials=1))])
def test_overlapped_back_to_back_shared_workspace(sk, dev, name, kw, tile, red):
    # Twelve calls over three input sets, one workspace, no synchronisation in between:
    # each call's flags, counters and partial tiles are reused by the next. Integer inputs
    # keep every sum exact, so the atomic reduction must match exactly too.
    M, N, K, sms = 768, 1024, 2048, 148
    sets = []
    for i in range(3):
        a, b = synth.small_int_inputs(M, N, K, "NN", 60 + i)
        sets.append((_bf16(a, dev), _bf16(b, dev)))
    stream = torch.cuda.current_stream(dev)

    def run(overlap):
        sched = sk.schedule(tile=tile, overlap=overlap, **kw)
        nbytes = sk.sk_workspace_size(M, N, K, sms, sched, red)
        ws = torch.zeros(nbytes, dtype=torch.uint8, device=dev)
        outs = [torch.full((M, N), U.SENTINEL, dtype=torch.float32, device=dev) for _ in range(12)]
        torch.cuda.synchronize(dev)
        for i, C in enumerate(outs):
            A, B = sets[i % 3]
            sk.sk_gemm(A, B, C, sk.SK_F32, M, N, K, sk.SK_NN, sched, red, sms, ws, nbytes, stream)
        assert sk.sk_status(ws, stream) == sk.SK_OK
        return [o.cpu().numpy() for o in outs]

    ref, got, early = run(0), run(1), run(2)
    for i in range(12):
        assert np.array_equal(got[i], ref[i % 3]), i
        assert np.array_equal(early[i], ref[i % 3]), i
        assert np.array_equal(ref[i], ref[i % 3]), i
    assert not np.array_equal(ref[0], ref[1])


@pytest.mark.parametrize("red", [DET, ATOM])
@pytest.mark.parametrize("tile", [0, 2])
@pytest.mark.parametrize("name,kw", [("hybrid", dict(mode=3)), ("streamk", dict(mode=2)),
                                     ("slabs2", dict(mode=1, splits=2, split_partials=1)),
                                     ("streamk_sep", dict(mode=2, split_partials=1))])
def test_early_operand_loads_one_output(sk, dev, name, kw, tile, red):
    # overlap = 2: eight calls over independent operands (integer, so every sum is exact)
    # write the same C one after another. Each call's epilogue must wait for the one before,
    # so C ends as the last call's product, and each intermediate product (copied out right
    # after its call) equals the non-overlapped result.
    M, N, K, sms = 768, 1024, 2048, 148
    sets = []
    for i in range(4):
        a, b = synth.small_int_inputs(M, N, K, "NN", 70 + i)
        sets.append((_bf16(a, dev), _bf16(b, dev)))
    stream = torch.cuda.current_stream(dev)

    def run(overlap, copy_out):
        sched = sk.schedule(tile=tile, overlap=overlap, **kw)
        nbytes = sk.sk_workspace_size(M, N, K, sms, sched, red)
        ws = torch.zeros(nbytes, dtype=torch.uint8, device=dev)
        C = torch.full((M, N), U.SENTINEL, dtype=torch.float32, device=dev)
        outs = []
        torch.cuda.synchronize(dev)
        for i in range(8):
            A, B = sets[i % 4]
            sk.sk_gemm(A, B, C, sk.SK_F32, M, N, K, sk.SK_NN, sched, red, sms, ws, nbytes, stream)
            if copy_out:
                outs.append(C.clone())
        assert sk.sk_status(ws, stream) == sk.SK_OK
        return C.cpu().numpy(), [o.cpu().numpy() for o in outs]

    ref_last, ref = run(0, True)
    last, _ = run(2, False)
    assert np.array_equal(last, ref[7])
    _, got = run(2, True)
    for i in range(8):
        assert np.array_equal(got[i], ref[i]), i
    assert not np.array_equal(ref[0], ref[1])


@pytest.mark.parametrize("tile", [0, 2])
def test_early_operand_loads_wait_limit(sk, dev, tile):
    # overlap = 2 behind a GEMM of about a hundred microseconds or more: the next calls'
    # first segments may start on SMs the long GEMM leaves free, long before it completes.
    # Their wait limits (50 us here) count from their own wait for it, so no call may
    # report a time-out, and every result is exact.
    Mb = Nb = 4096
    Kb = 8192
    big_a = torch.ones((Mb, Kb), dtype=torch.bfloat16, device=dev)
    big_b = torch.ones((Kb, Nb), dtype=torch.bfloat16, device=dev)
    big_c = torch.empty((Mb, Nb), dtype=torch.bfloat16, device=dev)
    M, N, K, sms = 512, 1024, 4096, 148
    sets = []
    for i in range(3):
        a, b = synth.small_int_inputs(M, N, K, "NN", 80 + i)
        sets.append((_bf16(a, dev), _bf16(b, dev)))
    stream = torch.cuda.current_stream(dev)
    big = sk.schedule(3, tile=2, overlap=1)
    nb_big = sk.sk_workspace_size(Mb, Nb, Kb, sms, big, DET)
    ws_big = torch.zeros(nb_big, dtype=torch.uint8, device=dev)

    def run(overlap):
        sched = sk.schedule(3, tile=tile, overlap=overlap)
        nbytes = sk.sk_workspace_size(M, N, K, sms, sched, DET)
        ws = torch.zeros(nbytes, dtype=torch.uint8, device=dev)
        outs = [torch.full((M, N), U.SENTINEL, dtype=torch.float32, device=dev) for _ in range(6)]
        torch.cuda.synchronize(dev)
        for i, C in enumerate(outs):
            if i % 3 == 0:
                sk.sk_gemm(big_a, big_b, big_c, sk.SK_BF16, Mb, Nb, Kb, sk.SK_NN, big, DET, sms, ws_big, nb_big,
                           stream)
            A, B = sets[i % 3]
            sk.sk_gemm_debug(A, B, C, sk.SK_F32, M, N, K, sk.SK_NN, sched, DET, sms, ws, nbytes, stream,
                             timeout_ns=50_000)
        assert sk.sk_status(ws, stream) == sk.SK_OK
        assert sk.sk_status(ws_big, stream) == sk.SK_OK
        return [o.cpu().numpy() for o in outs]

    got = run(2)
    ref = run(0)
    for i in range(6):
        assert np.array_equal(got[i], ref[i]), i
    assert np.all(big_c.float().cpu().numpy() == float(Kb))


@pytest.mark.parametrize("overlap", [1, 2])
def test_bench_configuration_back_to_back(sk, dev, overlap):
    # The wave-quantized GEMM (2048 x 2432 x 4096, BF16 out) in the configuration bench.py
    # times: hybrid rule on 148 SMs, 256 x 256 CTA pairs, overlapped launches back to back
    # over rotating input sets sharing one workspace. Three sets with different seeds, nine
    # launches; every output against the FP64 oracle on sampled rows, and outputs of the same
    # set equal bit for bit.
    from oracle import gemm as og
    base = synth.WAVEQ
    ws_ = [synth.Workload(base.name, base.M, base.N, base.K, base.layout, base.dist, seed, out=base.out)
           for seed in (base.seed, 31, 32)]
    bits = [synth.make_inputs(w) for w in ws_]
    sets = [(_bf16(a, dev), _bf16(b, dev)) for a, b in bits]
    M, N, K = base.M, base.N, base.K
    sched = sk.schedule(3, tile=2, overlap=overlap)
    nbytes = sk.sk_workspace_size(M, N, K, 148, sched, DET)
    ws = torch.zeros(nbytes, dtype=torch.uint8, device=dev)
    outs = [torch.full((M, N), U.SENTINEL, dtype=torch.bfloat16, device=dev) for _ in range(9)]
    stream = torch.cuda.current_stream(dev)
    torch.cuda.synchronize(dev)
    for i, C in enumerate(outs):
        A, B = sets[i % 3]
        sk.sk_gemm(A, B, C, sk.SK_BF16, M, N, K, sk.SK_NN, sched, DET, 148, ws, nbytes, stream)
    assert sk.sk_status(ws, stream) == sk.SK_OK
    got = [o.float().cpu().numpy().astype(np.float64) for o in outs]
    rows = U.sample_rows(M, 24, seed=5)
    for j, (a, b) in enumerate(bits):
        ref = og.ref_rows(a, b, base.layout, rows)
        U.assert_close(got[j][rows], ref, f"set {j}")
        for i in range(j + 3, 9, 3):
            assert np.array_equal(got[i], got[j]), (i, j)


def test_skinny_split_k_chain_independent_operands(sk, dev):
    # The skinny long-K shape (512 x 512 x 65536) as Split-K in 16 slabs with the reduction
    # pass, six launches over three input sets sharing one workspace. With overlap = 2 the
    # reduction runs on the 24 SMs the 128-CTA GEMM leaves idle and lets the next GEMM start
    # beside it; every result must equal the overlap = 1 chain bit for bit, and the first
    # three match the FP64 oracle on sampled rows.
    from oracle import gemm as og
    base = synth.SKINNY
    wl = [synth.Workload(base.name, base.M, base.N, base.K, base.layout, base.dist, seed, out=base.out)
          for seed in (base.seed, 61, 62)]
    bits = [synth.make_inputs(w) for w in wl]
    sets = [(_bf16(a, dev), _bf16(b, dev)) for a, b in bits]
    M, N, K = base.M, base.N, base.K
    stream = torch.cuda.current_stream(dev)

    def run(overlap):
        sched = sk.schedule(1, 16, split_partials=1, tile=2, overlap=overlap)
        nbytes = sk.sk_workspace_size(M, N, K, 148, sched, DET)
        ws = torch.zeros(nbytes, dtype=torch.uint8, device=dev)
        outs = [torch.full((M, N), U.SENTINEL, dtype=torch.bfloat16, device=dev) for _ in range(6)]
        torch.cuda.synchronize(dev)
        for i, C in enumerate(outs):
            A, B = sets[i % 3]
            sk.sk_gemm(A, B, C, sk.SK_BF16, M, N, K, sk.SK_NN, sched, DET, 148, ws, nbytes, stream)
        assert sk.sk_status(ws, stream) == sk.SK_OK
        return [o.float().cpu().numpy().astype(np.float64) for o in outs]

    ref, got = run(1), run(2)
    for i in range(6):
        assert np.array_equal(got[i], ref[i]), i
        assert np.array_equal(ref[i], ref[i % 3]), i
    rows = U.sample_rows(M, 12, seed=9)
    for j, (a, b) in enumerate(bits):
        U.assert_close(ref[j][rows], og.ref_rows(a, b, base.layout, rows), f"set {j}")
