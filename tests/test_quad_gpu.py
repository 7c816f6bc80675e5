"""The four-CTA tile (SK_TILE_256x512_QUAD): two CTA pairs side by side in a cluster of four,
sharing the A rows by TMA multicast. The same parity bar as the other shapes: against the
FP64 oracle, exactly on integer inputs, across data-parallel, Stream-K and the hybrid rule
with both reductions, on a small problem, ragged shapes, the full wave-quantized GEMM and
back-to-back overlapped launches; and the time-out path of its waits. A GB300 holds 36
clusters of four at once (144 SMs), so the full-size cases run on 144 SMs.
"""
import numpy as np
import pytest
import torch

import synth
from oracle import gemm as og

from . import gpu_util as U

pytestmark = pytest.mark.gpu

DET, ATOM = 0, 1
QUAD = 4
MODES = [("dp", 0), ("streamk", 2), ("hybrid", 3)]


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


@pytest.mark.parametrize("red", [DET, ATOM])
@pytest.mark.parametrize("name,mode", MODES)
def test_quad_toy(sk, dev, name, mode, red):
    # 128 x 640 x 256 on 4 units (16 CTAs): 2 tiles of 256 x 512 x 4 k-iterations, so
    # Stream-K splits both tiles across units and every reduction path runs.
    w = synth.TOY
    A_bits, B_bits = U.inputs(w)
    A, B = U.to_dev(A_bits, dev), U.to_dev(B_bits, dev)
    got, guards, _, status = U.gemm(sk, A, B, w.M, w.N, w.K, w.layout, sk.schedule(mode, units=4, tile=QUAD), red,
                                    16, w.out, dev)
    assert status == sk.SK_OK and guards
    assert not np.any(got == U.SENTINEL)
    U.assert_close(got, U.reference(w), name)


@pytest.mark.parametrize("layout", ["NN", "NT"])
@pytest.mark.parametrize("red", [DET, ATOM])
@pytest.mark.parametrize("sms", [8, 28, 144])
@pytest.mark.parametrize("name,mode", MODES)
def test_quad_integer_exact(sk, dev, name, mode, red, sms, layout):
    # Ragged in M, N and K (300 x 264 x 520 and 700 x 1000 x 1096): integer inputs keep every
    # partial sum exact, so the result must equal the oracle exactly, FP32 and BF16 out.
    for M, N, K in ((300, 264, 520), (700, 1000, 1096)):
        A_bits, B_bits = synth.small_int_inputs(M, N, K, layout, 23)
        A, B = U.to_dev(A_bits, dev), U.to_dev(B_bits, dev)
        ref = og.ref_gemm(A_bits, B_bits, layout)
        sched = sk.schedule(mode, tile=QUAD)
        got, guards, _, status = U.gemm(sk, A, B, M, N, K, layout, sched, red, sms, "f32", dev)
        assert status == sk.SK_OK and guards
        assert np.array_equal(got, ref), (M, N, K)
        got16, guards, _, status = U.gemm(sk, A, B, M, N, K, layout, sched, red, sms, "bf16", dev)
        assert status == sk.SK_OK and guards
        want16 = torch.from_numpy(ref.astype(np.float32)).to(torch.bfloat16).float().numpy()
        assert np.array_equal(got16, want16.astype(np.float64)), (M, N, K)


@pytest.mark.parametrize("red", [DET, ATOM])
@pytest.mark.parametrize("name,mode", MODES)
def test_quad_waveq_full(sk, dev, name, mode, red):
    # 2048 x 2432 x 4096 (40 tiles of 256 x 512 on 36 units at 144 SMs), BF16 out; full
    # comparison with the FP64 oracle.
    w = synth.WAVEQ
    A_bits, B_bits = U.inputs(w)
    A, B = U.to_dev(A_bits, dev), U.to_dev(B_bits, dev)
    got, guards, _, status = U.gemm(sk, A, B, w.M, w.N, w.K, w.layout, sk.schedule(mode, tile=QUAD), red, 144,
                                    w.out, dev)
    assert status == sk.SK_OK and guards
    U.assert_close(got, U.reference(w), name)


def test_quad_deterministic_repeats_and_overlap(sk, dev):
    # The hybrid rule on the wave-quantized GEMM: ten plain launches give the same bits, and
    # so do overlapped launches back to back sharing one workspace.
    w = synth.WAVEQ
    A_bits, B_bits = U.inputs(w)
    A, B = U.to_dev(A_bits, dev), U.to_dev(B_bits, dev)
    first, _, ws, status = U.gemm(sk, A, B, w.M, w.N, w.K, w.layout, sk.schedule(3, tile=QUAD), DET, 144, w.out, dev)
    assert status == sk.SK_OK
    for _ in range(9):
        again, _, _, status = U.gemm(sk, A, B, w.M, w.N, w.K, w.layout, sk.schedule(3, tile=QUAD), DET, 144, w.out,
                                     dev, ws)
        assert status == sk.SK_OK and np.array_equal(again, first)
    sched = sk.schedule(3, tile=QUAD, overlap=1)
    nb = sk.sk_workspace_size(w.M, w.N, w.K, 144, sched, DET)
    ws2 = torch.zeros(nb, dtype=torch.uint8, device=dev)
    outs = [torch.full((w.M, w.N), U.SENTINEL, dtype=torch.bfloat16, device=dev) for _ in range(6)]
    stream = torch.cuda.current_stream(dev)
    torch.cuda.synchronize(dev)
    for C in outs:
        sk.sk_gemm(A, B, C, sk.SK_BF16, w.M, w.N, w.K, sk.SK_NN, sched, DET, 144, ws2, nb, stream)
    assert sk.sk_status(ws2, stream) == sk.SK_OK
    for C in outs:
        assert np.array_equal(C.float().cpu().numpy().astype(np.float64), first)


@pytest.mark.parametrize("red", [DET, ATOM])
def test_quad_wait_timeout_reports_status(sk, dev, red):
    # Producers never raise their flags: the owners' waits (and with the deterministic
    # reduction the producer warp's flag wait for the ring copies) run out after 50 ms; the
    # status is SK_ETIMEOUT, and the workspace works again once zeroed.
    w = synth.TOY
    sched = sk.schedule(2, units=4, tile=QUAD)
    A_bits, B_bits = U.inputs(w)
    A, B = U.to_dev(A_bits, dev), U.to_dev(B_bits, dev)
    ws = U.new_workspace(sk, w.M, w.N, w.K, 16, sched, red, dev)
    _, _, _, status = U.gemm(sk, A, B, w.M, w.N, w.K, "NN", sched, red, 16, "f32", dev, ws,
                             skip_producer_signal=1, timeout_ns=50_000_000)
    assert status == sk.SK_ETIMEOUT
    ws[0].zero_()
    got, guards, _, status = U.gemm(sk, A, B, w.M, w.N, w.K, "NN", sched, red, 16, "f32", dev, ws)
    assert status == sk.SK_OK and guards
    U.assert_close(got, U.reference(w), "after time-out")


@pytest.mark.parametrize("name,mode", MODES)
def test_quad_overlapped_chain_equals_serial(sk, dev, name, mode):
    # Five dependent GEMMs X_{i+1} = X_i . W_i (640 x 768 x 768, BF16 out), launched back to
    # back with and without the overlapped launch: a missing wait for the previous kernel
    # would read X_i before it is written, so both chains must agree bit for bit.
    M, K = 640, 768
    X0 = U.to_dev(synth.make_inputs(synth.Workload("chain_x", M, K, K, seed=40))[0], dev)
    Ws = [U.to_dev(synth.make_inputs(synth.Workload("chain_w", K, K, K, seed=41 + i))[1], dev) for i in range(5)]
    stream = torch.cuda.current_stream(dev)

    def chain(overlap):
        sched = sk.schedule(mode, tile=QUAD, overlap=overlap)
        nb = sk.sk_workspace_size(M, K, K, 144, sched, DET)
        ws = torch.zeros(nb, dtype=torch.uint8, device=dev)
        outs = [torch.full((M, K), U.SENTINEL, dtype=torch.bfloat16, device=dev) for _ in Ws]
        x = X0
        torch.cuda.synchronize(dev)
        for W, Y in zip(Ws, outs):
            sk.sk_gemm(x, W, Y, sk.SK_BF16, M, K, K, sk.SK_NN, sched, DET, 144, ws, nb, stream)
            x = Y
        assert sk.sk_status(ws, stream) == sk.SK_OK
        return [y.float().cpu().numpy() for y in outs]

    ref, got = chain(0), chain(1)
    for i, (g, r) in enumerate(zip(got, ref)):
        assert not np.any(r == U.SENTINEL)
        assert np.array_equal(g, r), (name, i)
