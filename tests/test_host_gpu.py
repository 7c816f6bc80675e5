"""sk_gemm_host: GEMMs over host buffers through device staging sets.

Every problem's C must equal, bit for bit, sk_gemm on device copies of the same inputs with
the same schedule (the deterministic reduction does not depend on where the operands came
from), and match the FP64 oracle within the pass criteria. Covered: depth 1 (every copy and
GEMM in order on one stream) and depth 2 (two staging sets used in turn, uploads and
downloads on two more streams, so that problem i's buffers are reused by problem i + 2 while
other problems are in flight), page-locked and pageable host memory, overlapped launches,
Split-K slabs with the reduction pass, one C buffer shared by every problem, K == 0, and the
errors that need the device (nothing may be enqueued).
"""
import numpy as np
import pytest
import torch

import synth
from oracle import gemm as og

from . import gpu_util as U

pytestmark = pytest.mark.gpu

DET = 0
COUNT = 5


@pytest.fixture(scope="module")
def sk():
    import __graft_entry__ as ge
    ge.build()
    import gemm_work_decomposition_gb300 as m
    return m


def _host_bf16(bits: np.ndarray, pinned: bool) -> torch.Tensor:
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16).copy()).view(torch.bfloat16)
    return t.pin_memory() if pinned else t


def _problems(name, M, N, K, layout, dist, out, count):
    return [synth.Workload(f"{name}_{i}", M, N, K, layout, dist, 40 + i, out=out) for i in range(count)]


# (case, M, N, K, layout, dist, out, schedule kwargs, num_sms)
CASES = [
    ("hybrid_pair", 512, 768, 1024, "NN", "normal_sqrtk", "bf16", dict(mode=3, tile=2, overlap=1), 148),
    ("slabs_nt_overlap2", 96, 512, 2048, "NT", "normal", "f32", dict(mode=1, splits=4, split_partials=1, overlap=2),
     148),
    ("streamk_128_ragged", 200, 264, 712, "NN", "normal_sqrtk", "bf16", dict(mode=2, tile=0), 148),
]


def _run_host(sk, dev, ws, probs, sched, sms, depth, pinned, C_host, out, streams):
    w0 = probs[0]
    code = sk.SK_F32 if out == "f32" else sk.SK_BF16
    lay = sk.SK_NN if w0.layout == "NN" else sk.SK_NT
    nstage = sk.sk_host_staging_size(w0.M, w0.N, w0.K, code, depth)
    staging = torch.empty(nstage, dtype=torch.uint8, device=dev)
    A_h, B_h = [], []
    for w in probs:
        a, b = U.inputs(w)
        A_h.append(_host_bf16(a, pinned))
        B_h.append(_host_bf16(b, pinned))
    main, cin, cout = streams
    buf, nbytes = ws
    sk.sk_gemm_host(A_h, B_h, C_host, code, w0.M, w0.N, w0.K, lay, sched, DET, sms, staging, nstage, depth, buf,
                    nbytes, main, cin if depth == 2 else None, cout if depth == 2 else None)
    torch.cuda.synchronize(dev)
    assert sk.sk_status(buf, main) == sk.SK_OK


@pytest.mark.parametrize("pinned", [True, False], ids=["pinned", "pageable"])
@pytest.mark.parametrize("depth", [1, 2])
@pytest.mark.parametrize("case,M,N,K,layout,dist,out,kw,sms", CASES, ids=[c[0] for c in CASES])
def test_gemm_host_matches_device_gemm(sk, case, M, N, K, layout, dist, out, kw, sms, depth, pinned):
    dev = torch.device("cuda:0")
    probs = _problems(case, M, N, K, layout, dist, out, COUNT)
    sched = sk.schedule(**kw)
    ws = U.new_workspace(sk, M, N, K, sms, sched, DET, dev)
    dt = torch.float32 if out == "f32" else torch.bfloat16
    C_host = [torch.full((M, N), U.SENTINEL, dtype=dt) for _ in probs]
    if pinned:
        C_host = [c.pin_memory() for c in C_host]
    streams = (torch.cuda.current_stream(dev), torch.cuda.Stream(dev), torch.cuda.Stream(dev))
    _run_host(sk, dev, ws, probs, sched, sms, depth, pinned, C_host, out, streams)
    for w, c in zip(probs, C_host):
        a, b = U.inputs(w)
        want, guards_ok, _, status = U.gemm(sk, U.to_dev(a, dev), U.to_dev(b, dev), M, N, K, layout, sched, DET, sms,
                                           out, dev, ws=ws)
        assert guards_ok and status == sk.SK_OK
        got = c.float().numpy().astype(np.float64)
        assert np.array_equal(got, want), w.name
        U.assert_close(got, og.ref_gemm(a, b, layout), w.name)


def test_gemm_host_one_output_buffer_and_repeat_calls(sk):
    # Every problem writes the same host C: the downloads run in problem order, so the last
    # problem's result stays. A second call reuses the staging sets and the workspace.
    dev = torch.device("cuda:0")
    case, M, N, K, layout, dist, out, kw, sms = CASES[0]
    probs = _problems("shared_c", M, N, K, layout, dist, out, 3)
    sched = sk.schedule(**kw)
    ws = U.new_workspace(sk, M, N, K, sms, sched, DET, dev)
    c = torch.full((M, N), U.SENTINEL, dtype=torch.bfloat16).pin_memory()
    streams = (torch.cuda.Stream(dev), torch.cuda.Stream(dev), torch.cuda.Stream(dev))
    for _ in range(2):
        c.fill_(U.SENTINEL)
        _run_host(sk, dev, ws, probs, sched, sms, 2, True, [c, c, c], out, streams)
        a, b = U.inputs(probs[-1])
        want, _, _, _ = U.gemm(sk, U.to_dev(a, dev), U.to_dev(b, dev), M, N, K, layout, sched, DET, sms, out, dev,
                               ws=ws)
        assert np.array_equal(c.float().numpy().astype(np.float64), want)


def test_gemm_host_k_zero(sk):
    dev = torch.device("cuda:0")
    M, N = 136, 256
    sched = sk.schedule(sk.SK_HYBRID)
    ws = U.new_workspace(sk, M, N, 64, 148, sched, DET, dev)
    nstage = sk.sk_host_staging_size(M, N, 0, sk.SK_F32, 2)
    staging = torch.empty(nstage, dtype=torch.uint8, device=dev)
    C_host = [torch.full((M, N), U.SENTINEL).pin_memory() for _ in range(3)]
    s = [torch.cuda.Stream(dev) for _ in range(3)]
    sk.sk_gemm_host([0] * 3, [0] * 3, C_host, sk.SK_F32, M, N, 0, sk.SK_NN, sched, DET, 148, staging, nstage, 2,
                    ws[0], ws[1], s[0], s[1], s[2])
    torch.cuda.synchronize(dev)
    assert all(bool((c == 0).all()) for c in C_host)


def test_gemm_host_device_errors_enqueue_nothing(sk):
    dev = torch.device("cuda:0")
    M, N, K = 512, 768, 1024
    w = _problems("errors", M, N, K, "NN", "normal_sqrtk", "bf16", 1)[0]
    a, b = U.inputs(w)
    A_h, B_h = [_host_bf16(a, True)], [_host_bf16(b, True)]
    C_h = [torch.full((M, N), U.SENTINEL, dtype=torch.bfloat16).pin_memory()]
    nstage = sk.sk_host_staging_size(M, N, K, sk.SK_BF16, 1)
    staging = torch.empty(nstage, dtype=torch.uint8, device=dev)
    stream = torch.cuda.Stream(dev)
    good = sk.schedule(sk.SK_HYBRID, tile=2)
    ws, nbytes = U.new_workspace(sk, M, N, K, 148, good, DET, dev)
    too_many = sk.schedule(sk.SK_STREAMK, units=4096, tile=2)  # more CTA pairs than the device holds
    nws = sk.sk_workspace_size(M, N, K, 148, too_many, DET)
    ws_big = torch.zeros(nws, dtype=torch.uint8, device=dev)
    for sched, buf, size, code in [(good, ws, nbytes - 256, sk.SK_EWORKSPACE),
                                   (too_many, ws_big, nws, sk.SK_ERESIDENCY)]:
        with pytest.raises(sk.SkError) as e:
            sk.sk_gemm_host(A_h, B_h, C_h, sk.SK_BF16, M, N, K, sk.SK_NN, sched, DET, 148, staging, nstage, 1, buf,
                            size, stream)
        assert e.value.code == code
    torch.cuda.synchronize(dev)
    assert bool((C_h[0].float() == U.SENTINEL).all())


def test_gemm_host_atomic_reduction(sk):
    # FP32 atomics: the bits may depend on arrival order, so only the tolerance is checked.
    dev = torch.device("cuda:0")
    M, N, K, sms = 256, 640, 1024, 148
    probs = _problems("atomic", M, N, K, "NN", "uniform", "f32", 3)
    sched = sk.schedule(sk.SK_STREAMK)
    nbytes = sk.sk_workspace_size(M, N, K, sms, sched, sk.SK_ATOMIC)
    ws = torch.zeros(nbytes, dtype=torch.uint8, device=dev)
    nstage = sk.sk_host_staging_size(M, N, K, sk.SK_F32, 2)
    staging = torch.empty(nstage, dtype=torch.uint8, device=dev)
    A_h, B_h = [], []
    for w in probs:
        a, b = U.inputs(w)
        A_h.append(_host_bf16(a, True))
        B_h.append(_host_bf16(b, True))
    C_h = [torch.full((M, N), U.SENTINEL).pin_memory() for _ in probs]
    s = [torch.cuda.Stream(dev) for _ in range(3)]
    sk.sk_gemm_host(A_h, B_h, C_h, sk.SK_F32, M, N, K, sk.SK_NN, sched, sk.SK_ATOMIC, sms, staging, nstage, 2,
                    ws, nbytes, s[0], s[1], s[2])
    torch.cuda.synchronize(dev)
    assert sk.sk_status(ws, s[0]) == sk.SK_OK
    for w, c in zip(probs, C_h):
        a, b = U.inputs(w)
        U.assert_close(c.numpy().astype(np.float64), og.ref_gemm(a, b, "NN"), w.name)
