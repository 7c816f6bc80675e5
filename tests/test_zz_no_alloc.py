"""sk_gemm_noalloc: the GEMM for callers that cannot allocate device memory.

Plug-ins whose host application owns every device allocation, processes held to a memory
budget fixed at start-up, and loops where cudaMalloc / cudaFree would synchronise the
device cannot hand sk_gemm a workspace of their own. sk_gemm_noalloc uses a scratch array
owned by the library instead. This test calls it through the C ABI twice in a row and
checks each result against sk_gemm with a caller-owned workspace, within the same
tolerance the other GPU tests use (and bit for bit, since the deterministic reduction
does not depend on where the workspace lives). It must pass alone in a fresh process and
after the other tests, so it lives in a file that pytest collects last.
"""
import ctypes

import numpy as np
import pytest
import torch

import synth

from . import gpu_util as U

pytestmark = pytest.mark.gpu


def _noalloc(sk, A, B, C, code, w, sched, red, sms, stream):
    L = sk.lib()
    return L.sk_gemm_noalloc(A.data_ptr(), B.data_ptr(), C.data_ptr(), code, w.M, w.N, w.K,
                             sk.SK_NN if w.layout == "NN" else sk.SK_NT, sched, red, sms,
                             ctypes.c_void_p(stream.cuda_stream))


def test_noalloc_matches_sk_gemm_twice():
    import __graft_entry__ as ge
    ge.build()
    import gemm_work_decomposition_gb300 as sk
    dev = torch.device("cuda:0")
    stream = torch.cuda.current_stream(dev)
    cases = [
        # (workload, schedule, reduction, units): wave-quantized hybrid on 148 SMs; the toy
        # Stream-K case with atomic reduction on 4 units; small-M Split-K slabs summed by the
        # reduction pass (split_partials 1) and inside the launch (2); Stream-K merged by the
        # separate fixup pass (split_partials 1), whose workspace has the slot layout.
        (synth.WAVEQ, sk.schedule(sk.SK_HYBRID), sk.SK_DETERMINISTIC, 148),
        (synth.TOY, sk.schedule(sk.SK_STREAMK, units=4), sk.SK_ATOMIC, 4),
        (synth.SMALLM_96, sk.schedule(sk.SK_SPLITK, splits=8, split_partials=1), sk.SK_DETERMINISTIC, 148),
        (synth.SMALLM_96, sk.schedule(sk.SK_SPLITK, splits=4, split_partials=2), sk.SK_DETERMINISTIC, 148),
        (synth.TOY, sk.schedule(sk.SK_STREAMK, units=4, split_partials=1), sk.SK_DETERMINISTIC, 4),
        (synth.SMALLM_256, sk.schedule(sk.SK_STREAMK, units=40, split_partials=1), sk.SK_DETERMINISTIC, 148),
    ]
    for call, (w, sched, red, sms) in enumerate(cases * 2):
        A_bits, B_bits = U.inputs(w)
        A, B = U.to_dev(A_bits, dev), U.to_dev(B_bits, dev)
        want, guards, _, status = U.gemm(sk, A, B, w.M, w.N, w.K, w.layout, sched, red, sms, w.out, dev)
        assert status == sk.SK_OK and guards
        dt = torch.float32 if w.out == "f32" else torch.bfloat16
        code = sk.SK_F32 if w.out == "f32" else sk.SK_BF16
        C = torch.full((w.M * w.N + U.N_GUARD,), U.SENTINEL, dtype=dt, device=dev)
        C[w.M * w.N:] = U.GUARD
        assert _noalloc(sk, A, B, C, code, w, sched, red, sms, stream) == sk.SK_OK
        torch.cuda.synchronize(dev)
        host = C.float().cpu().numpy().astype(np.float64)
        assert np.all(host[w.M * w.N:] == U.GUARD)
        got = host[:w.M * w.N].reshape(w.M, w.N)
        U.assert_close(got, want, f"call {call}")
        U.assert_close(got, U.reference(w), f"call {call} vs oracle")
        if red == sk.SK_DETERMINISTIC:
            assert np.array_equal(got, want)
    # A problem whose workspace exceeds the fixed scratch is rejected before any work.
    w = synth.WAVEQ
    big = sk.schedule(sk.SK_SPLITK, splits=2)
    assert sk.sk_workspace_size(w.M, w.N, w.K, 148, big, 0) > sk.SK_NOALLOC_SCRATCH_BYTES
    A = torch.zeros(16, dtype=torch.bfloat16, device=dev)
    C = torch.zeros(16, dtype=torch.bfloat16, device=dev)
    assert _noalloc(sk, A, A, C, sk.SK_BF16, w, big, 0, 148, stream) == sk.SK_EWORKSPACE
