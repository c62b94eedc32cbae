"""The bounded waits that guard the tensor-core kernels end on their own.

Every mbarrier wait in the GEMM kernels gives up after a limit and the launch
reports FP4_ERR_TIMEOUT in its status word instead of hanging. fp4_wait_selftest
runs one such wait on a barrier that nothing arrives on (no fault, no trap, no
endless loop): the kernel must end within its limit, set the status, and leave the
CUDA context usable for the next call.
"""
import time

import numpy as np
import pytest

import block_scaled_fp4_mx_gb300 as fp4
from block_scaled_fp4_mx_gb300 import inputs

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


@pytest.mark.parametrize("mode", [0, 1])
def test_wait_gives_up_and_reports_timeout(mode):
    """Spinning (mode 0) and sleeping (mode 1) waits: the status word says
    ERR_TIMEOUT, the kernel ends within a few seconds, the context still works."""
    torch.cuda.synchronize()
    t0 = time.monotonic()
    status = fp4.fp4_wait_selftest(mode, device="cuda:0")
    torch.cuda.synchronize()
    elapsed = time.monotonic() - t0
    assert int(status.item()) == fp4.Status.ERR_TIMEOUT
    assert elapsed < 5.0, elapsed
    # the context is usable: an unpack right after gives the expected bits
    w = inputs.mx_random(8, 64, seed=3)
    p = torch.from_numpy(w.packed).to("cuda:0")
    s = torch.from_numpy(w.scales).to("cuda:0")
    out = fp4.fp4_mx_unpack(p, s)
    torch.cuda.synchronize()
    again = fp4.fp4_mx_unpack(p, s)
    assert torch.equal(out.view(torch.int16), again.view(torch.int16))


def test_completed_wait_leaves_status_alone():
    status = torch.zeros(1, dtype=torch.int32, device="cuda:0")
    fp4.fp4_wait_selftest(2, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
