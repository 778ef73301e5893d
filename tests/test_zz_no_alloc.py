"""kda_bwd_noalloc: the backward for callers that cannot allocate device memory.

Callers such as code running under a framework's own memory pool, a server that
has carved up the GPU in advance, or a plug-in host that forbids allocation
cannot hand the library a context workspace. kda_bwd_noalloc takes only their
inputs and outputs and keeps every intermediate in a fixed array inside the
library. This file checks, through the C ABI, that two calls in a row (with
different inputs, so stale scratch contents would show) give the gradients of
the FP64 oracle and of the regular kda_fwd + kda_bwd pair within the
tolerances of the parity tests, that the status word reads back clean after a
good call and flags a device cu_seqlens that disagrees with its host mirror,
and that a problem larger than the array is refused with a clear error. It is
named so that pytest collects it last.
"""

import pytest
import torch

import kda_inputs as ki
from kda_test_utils import OUT_NAMES, compare, run_gpu, run_oracle, to_device

pytestmark = pytest.mark.gpu

GRADS = OUT_NAMES[2:]


@pytest.fixture(scope="module", autouse=True)
def library():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    from linear_attention_gated_gb300 import build
    build.build()
    from linear_attention_gated_gb300 import kda
    kda.load_library()


def _noalloc(x, d=None):
    from linear_attention_gated_gb300 import kda_bwd_noalloc
    d = to_device(x) if d is None else d
    grads = kda_bwd_noalloc(d["q"], d["k"], d["v"], d["g"], d["beta"], d["A_log"], d["dt_bias"], d["h0"],
                            d["do"], d["dfinal_state"], cu_seqlens=d.get("cu_seqlens"),
                            cu_seqlens_cpu=d.get("cu_seqlens_cpu"))
    torch.cuda.synchronize()
    return dict(zip(GRADS, (t.cpu() for t in grads)))


def _as_ref(gpu):
    return {k: v.double().numpy() for k, v in gpu.items()}


def test_two_calls_match_oracle_and_regular_backward():
    from linear_attention_gated_gb300 import noalloc_status
    # packed ragged with GQA 1:2, then a fixed layout with equal heads
    cases = [ki.make_inputs(1, 0, 2, 4, seed=21, lengths=[100, 37, 260]),
             ki.make_inputs(2, 150, 3, 3, seed=22)]
    for x in cases:
        got = _noalloc(x)
        noalloc_status()
        compare(got, run_oracle(x), names=GRADS)
        reg, _ = run_gpu(x)
        compare(got, _as_ref({k: reg[k] for k in GRADS}), names=GRADS)


def test_device_offsets_that_disagree_with_the_mirror_are_reported():
    from linear_attention_gated_gb300 import KdaError, noalloc_status
    x = ki.make_inputs(1, 0, 1, 2, seed=24, lengths=[40, 60])
    d = to_device(x)
    d["cu_seqlens"] = torch.tensor([0, 40, 90], dtype=torch.int64, device="cuda")  # ends short of T = 100
    _noalloc(x, d)
    with pytest.raises(KdaError) as e:
        noalloc_status()
    assert e.value.name == "KDA_ERR_INVALID_ARGUMENT"
    assert "cu_seqlens" in str(e.value)
    # the next good call clears the word
    got = _noalloc(x)
    noalloc_status()
    compare(got, run_oracle(x), names=GRADS)


def test_too_large_problem_is_refused():
    from linear_attention_gated_gb300 import KdaError
    x = ki.make_inputs(1, 4096, 1, 16, seed=23)
    with pytest.raises(KdaError) as e:
        _noalloc(x)
    assert e.value.name == "KDA_ERR_WORKSPACE_TOO_SMALL"
    assert "scratch" in str(e.value)
