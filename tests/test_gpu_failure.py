"""Failure detection on the GPU without a fault: a kernel's bounded wait on
an mbarrier phase that nothing completes, or on a flag word that nothing
sets, gives up after its limit, sets the library's sticky status word, and
the host reads REPOPS_ERR_TIMEOUT from it; the context stays usable (the next
GEMM is bit-exact and the status clean).  No trap, no assert, no bad
address: the wait simply runs out."""
import numpy as np
import pytest
import torch

from verifiable_repops_gemm_gb300 import inputs

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
REPOPS_ERR_TIMEOUT = -5


def test_bounded_wait_times_out_and_the_context_survives(rp, orc):
    L = rp.load()
    assert rp.device_status() == 0
    torch.cuda.synchronize()
    s = torch.cuda.current_stream()
    assert L.repops_selftest_bounded_wait(20_000_000, s.cuda_stream) == 0      # 20 ms limit
    assert rp.device_status() == REPOPS_ERR_TIMEOUT
    assert rp.device_status() == 0                                             # read and cleared
    A = inputs.normal((130, 70), 1.0, 1, DEV)
    B = inputs.normal((70, 90), 1.0, 2, DEV)
    C = rp.gemm(A, B)
    want = orc.gemm(A.cpu().numpy(), B.cpu().numpy())
    assert np.array_equal(C.cpu().numpy().view(np.uint32), want.view(np.uint32))
    assert rp.device_status() == 0


def test_flag_wait_times_out_and_the_context_survives(rp, orc):
    # the chained split's kind of wait (acquire loads of a flag another worker
    # releases): on a flag that nothing sets it gives up, the host reads the
    # timeout, and the next chained-split GEMM on the same context is
    # bit-exact with a clean status
    L = rp.load()
    torch.cuda.synchronize()
    assert rp.device_status() == 0
    s = torch.cuda.current_stream()
    assert L.repops_selftest_bounded_flag_wait(20_000_000, s.cuda_stream) == 0   # 20 ms limit
    assert rp.device_status() == REPOPS_ERR_TIMEOUT
    assert rp.device_status() == 0
    A = inputs.normal((300, 260), 1.0, 3, DEV)
    B = inputs.normal((260, 1000), 1.0, 4, DEV)
    C = rp.gemm_chained(A, B, config=4, workers=5)
    want = orc.gemm(A.cpu().numpy(), B.cpu().numpy())
    assert np.array_equal(C.cpu().numpy().view(np.uint32), want.view(np.uint32))
    assert rp.device_status() == 0


def test_status_word_scoped_per_caller(rp, orc):
    # A timeout on one caller's stream is reported in that caller's own word:
    # another caller's GEMM on another stream, bound to a word of its own, reads
    # status 0, and the shared word stays clean for callers that bound nothing.
    import threading
    L = rp.load()
    torch.cuda.synchronize()
    assert rp.device_status() == 0
    word_a = torch.zeros(1, dtype=torch.int32, device=DEV)
    word_b = torch.zeros(1, dtype=torch.int32, device=DEV)
    sa, sb = torch.cuda.Stream(), torch.cuda.Stream()
    A = inputs.normal((300, 200), 1.0, 11, DEV)
    B = inputs.normal((200, 260), 1.0, 12, DEV)
    torch.cuda.synchronize()
    out = {}

    def caller_a():
        rp.set_thread_status_word(word_a)
        assert L.repops_selftest_bounded_wait(50_000_000, sa.cuda_stream) == 0    # 50 ms limit
        out["a"] = rp.device_status(sa)
        rp.set_thread_status_word(None)

    def caller_b():
        rp.set_thread_status_word(word_b)
        with torch.cuda.stream(sb):
            out["C"] = rp.gemm(A, B, stream=sb)
        out["b"] = rp.device_status(sb)
        rp.set_thread_status_word(None)

    ta, tb = threading.Thread(target=caller_a), threading.Thread(target=caller_b)
    ta.start(); tb.start()
    ta.join(); tb.join()
    assert out["a"] == REPOPS_ERR_TIMEOUT
    assert out["b"] == 0
    assert rp.device_status() == 0                       # the shared word saw nothing
    torch.cuda.synchronize()
    assert int(word_a.item()) == 0 and int(word_b.item()) == 0   # both read and cleared
    want = orc.gemm(A.cpu().numpy(), B.cpu().numpy())
    assert np.array_equal(out["C"].cpu().numpy().view(np.uint32), want.view(np.uint32))
    # on one host thread, rebinding between calls scopes them the same way
    rp.set_thread_status_word(word_a)
    assert L.repops_selftest_bounded_wait(20_000_000, sa.cuda_stream) == 0
    rp.set_thread_status_word(word_b)
    rp.gemm(A, B, stream=sb)
    rp.set_thread_status_word(None)
    torch.cuda.synchronize()
    assert int(word_a.item()) == 1 and int(word_b.item()) == 0
    assert rp.device_status() == 0
