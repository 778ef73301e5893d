"""Training steps from and to host memory (kda_step_host) through the C ABI.

A step copies its host inputs into a device arena, runs the same forward and
backward as kda_fwd / kda_bwd and copies the outputs back, so its results must
be identical to the device-buffer calls, which the parity tests hold against
the FP64 oracle. Two arenas on two streams taken in turn (the overlapped
pipeline) must give the same results step after step.
"""

import pytest
import torch

import kda_inputs as ki
from kda_test_utils import OUT_NAMES, run_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def library():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    from linear_attention_gated_gb300 import build
    build.build()
    from linear_attention_gated_gb300 import kda
    kda.load_library()


IN_KEYS = ("q", "k", "v", "g", "beta", "A_log", "dt_bias", "h0", "do", "dfinal_state")


def _host_inputs(x):
    # the caller keeps these alive until the step's stream is synchronised: the
    # copies read them asynchronously
    return [x[k].contiguous().pin_memory() for k in IN_KEYS]


@pytest.mark.parametrize("case", ["fixed", "packed_gqa"])
def test_host_step_equals_device_calls(case):
    from linear_attention_gated_gb300 import HostStep
    if case == "fixed":
        x = ki.make_inputs(2, 80, 2, 2, seed=51)
    else:
        x = ki.make_inputs(1, 0, 2, 4, seed=52, lengths=[33, 70, 9])
    want, _ = run_gpu(x)
    B, T, Hqk = x["q"].shape[:3]
    step = HostStep(B, T, Hqk, x["v"].shape[2], cu_seqlens_cpu=x["cu_seqlens"])
    ins = _host_inputs(x)
    out = step(*ins, out=step.empty_outputs())
    step.synchronize()
    step.status()
    for name, got in zip(OUT_NAMES, out):
        assert torch.equal(got, want[name].cpu()), name


def test_two_arenas_in_turn():
    """Six steps alternating two arenas on shared copy-in, compute and copy-out
    streams; every step's outputs are the single-call results (the inputs change
    between steps, so a copy that overtook the kernels it must wait for would
    show)."""
    from linear_attention_gated_gb300 import HostStep
    lengths = [50, 17]
    xs = [ki.make_inputs(1, 0, 1, 2, seed=60 + i, lengths=lengths) for i in range(6)]
    wants = [run_gpu(x)[0] for x in xs]
    B, T, Hqk = xs[0]["q"].shape[:3]
    streams = [torch.cuda.Stream() for _ in range(3)]
    steps = [HostStep(B, T, Hqk, 2, cu_seqlens_cpu=xs[0]["cu_seqlens"], stream=streams[0], h2d_stream=streams[1],
                      d2h_stream=streams[2]) for _ in range(2)]
    outs, held = [], []
    for i, x in enumerate(xs):
        s = steps[i % 2]
        held.append(_host_inputs(x))
        outs.append(s(*held[-1], out=s.empty_outputs()))
    for s in steps:
        s.synchronize()
        s.status()
    for want, out in zip(wants, outs):
        for name, got in zip(OUT_NAMES, out):
            assert torch.equal(got, want[name].cpu()), name


def test_host_step_rejects_device_buffers():
    from linear_attention_gated_gb300 import HostStep, kda
    x = ki.make_inputs(1, 32, 1, 1, seed=53)
    step = HostStep(1, 32, 1, 1)
    ins = _host_inputs(x)
    with pytest.raises(ValueError, match="host tensor"):
        step(*[t.cuda() if i == 0 else t for i, t in enumerate(ins)], out=step.empty_outputs())
    # the C ABI itself refuses device memory where a host buffer is expected
    lib = kda.load_library()
    import ctypes
    dq = torch.empty_like(x["q"], device="cuda")
    out = list(step.empty_outputs())
    ptrs = [kda._ptr(t) for t in ins]
    rc = lib.kda_step_host(*ptrs[:8], None, 0, 1, 32, 1, 1, 128, float("nan"), -5.0, ptrs[8], ptrs[9],
                           kda._ptr(out[0]), kda._ptr(out[1]), kda._ptr(dq), *[kda._ptr(t) for t in out[3:]],
                           kda._ptr(step.arena), step.arena.numel(), ctypes.byref(step.handle),
                           ctypes.c_void_p(step.stream.cuda_stream), None, None)
    assert rc == 1 and b"host buffers" in lib.kda_last_error_message()
    small = torch.empty(1024, dtype=torch.uint8, device="cuda")
    rc = lib.kda_step_host(*ptrs[:8], None, 0, 1, 32, 1, 1, 128, float("nan"), -5.0, ptrs[8], ptrs[9],
                           *[kda._ptr(t) for t in out], kda._ptr(small), small.numel(),
                           ctypes.byref(step.handle), ctypes.c_void_p(step.stream.cuda_stream), None, None)
    assert rc == 7
