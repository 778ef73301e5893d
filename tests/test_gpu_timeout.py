"""Failure detection without a GPU fault: every wait in the kernels is bounded,
and a wait that runs out makes the kernel record a timeout in a device status
word that the host reads (KDA_ERR_DEVICE_TIMEOUT), leaving the context usable.

kda_selftest_device_timeout launches one CTA whose mbarrier wait nothing can
complete; the same bounded wait the kernels use gives up after about 1 ms. The
test checks the status it returns, then that a forward + backward on the same
device still matches the oracle.
"""

import time

import pytest
import torch

import kda_inputs as ki
from kda_test_utils import compare, run_gpu, run_oracle

pytestmark = pytest.mark.gpu

KDA_ERR_DEVICE_TIMEOUT = 6


@pytest.fixture(scope="module", autouse=True)
def library():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    from linear_attention_gated_gb300 import build
    build.build()
    from linear_attention_gated_gb300 import kda
    kda.load_library()


def test_bounded_wait_reports_timeout_and_device_stays_usable():
    from linear_attention_gated_gb300 import kda
    t0 = time.perf_counter()
    rc = kda.selftest_device_timeout()
    elapsed = time.perf_counter() - t0
    assert rc == KDA_ERR_DEVICE_TIMEOUT, (rc, kda.load_library().kda_last_error_message())
    assert elapsed < 5.0  # the wait gives up after ~1 ms of SM clock, not at a host timeout
    x = ki.make_inputs(1, 0, 1, 2, seed=21, lengths=[40, 17])
    gpu, _ = run_gpu(x)
    compare(gpu, run_oracle(x))
