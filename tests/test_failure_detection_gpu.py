"""Failure detection on the GPU without a fault.

Every wait in the library's kernels is bounded; one that runs out sets a device
status word, the kernel returns, and wg_check_status reports
WG_ERR_DEVICE_TIMEOUT.  The self-test entry point launches one thread waiting on
an mbarrier that nothing completes (a flag nothing sets).  The test checks that
the status is reported and cleared, and that the context stays usable: a normal
call afterwards runs and reports no error.
"""
import time

import numpy as np
import pytest

from implicit_gemm_gb300 import binding, build
from tests.common import make_inputs, spec

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    assert torch.cuda.is_available(), "the gpu tests need a CUDA device"
    build.build()
    binding.load()


def test_wait_that_runs_out_is_reported_and_context_survives():
    binding.wg_check_status()  # start clean
    t0 = time.time()
    binding.wg_selftest_timeout()
    with pytest.raises(binding.WgradError) as e:
        binding.wg_check_status()
    assert e.value.status == 6  # WG_ERR_DEVICE_TIMEOUT
    assert 1.0 < time.time() - t0 < 30.0  # the wait's limit, then the kernel returned
    binding.wg_check_status()  # the word was cleared
    # The context is usable: a normal call runs and matches a second one bit for bit.
    sp = spec(2, 1, 2, 16, 16, [9, 9], [3, 3], [1, 1], [1, 1], [1, 1], [1, 1])
    x, dy = make_inputs(sp, ("int", -2, 2), 71, 72)
    xd = torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).view(torch.bfloat16).cuda()
    dyd = torch.from_numpy(np.ascontiguousarray(dy).view(np.int16)).view(torch.bfloat16).cuda()
    a = binding.conv_bwd_weight(sp, xd, dyd, 3, "deterministic")
    b = binding.conv_bwd_weight(sp, xd, dyd, 3, "deterministic")
    binding.wg_check_status()
    assert torch.equal(a, b)
