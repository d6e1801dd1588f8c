"""Failure detection on the GPU without a fault: a kernel's bounded wait on
an mbarrier phase that nothing completes gives up after its limit, sets the
library's sticky status word, and the host reads REPOPS_ERR_TIMEOUT from it;
the context stays usable (the next GEMM is bit-exact and the status clean).
No trap, no assert, no bad address: the wait simply runs out."""
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
