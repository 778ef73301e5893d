"""The standalone backward with a caller-owned workspace
(flashinfer.kda_backward.recurrent_kda_backward: signature, description and the
parameters ``workspace`` and ``out``), compared with the FP64 oracle element by
element through the C ABI binding; workspace reuse, CUDA-graph capture after the
eager warm-up call, and the aliasing rule for the workspace."""

import pytest
import torch

import kda_inputs as ki
from kda_test_utils import OUT_NAMES, compare, run_oracle, to_device

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


def _call(d, workspace=None, out=None):
    from linear_attention_gated_gb300 import recurrent_kda_backward
    return recurrent_kda_backward(d["q"], d["k"], d["v"], d["g"], d["beta"], d["A_log"], d["dt_bias"], d["h0"],
                                  d["do"], d["dfinal_state"], cu_seqlens=d.get("cu_seqlens"),
                                  workspace=workspace, out=out, cu_seqlens_cpu=d.get("cu_seqlens_cpu"))


def _cpu(grads):
    return {k: t.cpu() for k, t in zip(GRADS, grads)}


def test_packed_ragged_gqa_matches_oracle():
    # GQA 1:4, four packed sequences of ragged, non-16-aligned lengths
    x = ki.make_inputs(1, 0, 2, 8, seed=31, lengths=[129, 17, 64, 250])
    got = _cpu(_call(to_device(x)))
    torch.cuda.synchronize()
    compare(got, run_oracle(x), names=GRADS)


def test_fixed_layout_matches_oracle():
    x = ki.make_inputs(2, 77, 3, 3, seed=32)
    got = _cpu(_call(to_device(x)))
    compare(got, run_oracle(x), names=GRADS)


def test_workspace_reuse_two_calls():
    from linear_attention_gated_gb300 import RecurrentKDABackwardWorkspace
    lengths = [100, 37, 91]
    xs = [ki.make_inputs(1, 0, 1, 2, seed=s, lengths=lengths) for s in (33, 34)]
    cu = xs[0]["cu_seqlens"]
    ws = RecurrentKDABackwardWorkspace(1, sum(lengths), 1, 2, cu_seqlens_cpu=cu)
    for x in xs:
        got = _cpu(_call(to_device(x), workspace=ws))
        compare(got, run_oracle(x), names=GRADS)
    ws.status()


def test_graph_capture_after_warm_up():
    from linear_attention_gated_gb300 import RecurrentKDABackwardWorkspace
    lengths = [70, 33]
    x0 = ki.make_inputs(1, 0, 2, 4, seed=35, lengths=lengths)
    x1 = ki.make_inputs(1, 0, 2, 4, seed=36, lengths=lengths)
    d = to_device(x0)
    ws = RecurrentKDABackwardWorkspace(1, sum(lengths), 2, 4, cu_seqlens_cpu=x0["cu_seqlens"])
    stream = torch.cuda.Stream()
    stream.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        # eager warm-up on the capture stream: the handle is bound to it from here on
        out = tuple(torch.empty_like(t) for t in _call(d, workspace=ws))
        _call(d, workspace=ws, out=out)
        stream.synchronize()
        with torch.cuda.graph(graph, stream=stream):
            _call(d, workspace=ws, out=out)
    # replay on new inputs copied into the captured buffers
    d1 = to_device(x1)
    for key in ("q", "k", "v", "g", "beta", "A_log", "dt_bias", "h0", "do", "dfinal_state"):
        d[key].copy_(d1[key])
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        graph.replay()
    torch.cuda.synchronize()
    replayed = {k: t.clone().cpu() for k, t in zip(GRADS, out)}
    with torch.cuda.stream(stream):
        eager = _cpu(_call(d, workspace=ws))
        torch.cuda.synchronize()
    for k in GRADS:
        assert torch.equal(replayed[k], eager[k]), k
    compare(replayed, run_oracle(x1), names=GRADS)
